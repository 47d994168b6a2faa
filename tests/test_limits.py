"""GPU parity at the limits of the entry points.

* The most groups a call takes (MSLKB_MAX_GROUPS = 1024, whose per-group tables the kernels
  keep in shared memory), on every layout and every kernel variant that serves it, with
  empty, one-row and clamped groups among them; whole outputs against the oracle.
* Operands and outputs of more than 2^31 elements (the sizes the host accepts go up to 2^40
  elements per operand): rows whose first element of A, of B or of the output lies past
  2^31 are compared in full against the oracle, so an element offset computed in 32 bits
  anywhere (loads, the cp.async loader, scales, direct and TMA stores) would show.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import random_codes
from parity_util import abs_codes, bits_of, compare

pytestmark = pytest.mark.gpu

G_MAX = 1024
TWO31 = 1 << 31


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fxbuild.build()
    fx.lib()


@pytest.fixture(scope="module")
def orc():
    return oracle.load(0)


@pytest.fixture(autouse=True)
def _fresh_status():
    fx.device_status()   # each test reads the bits its own calls set


def _names(prefix, exclude=()):
    try:
        fxbuild.build()
        names = [fx.variant_name(i) for i in range(fx.mslkb_num_variants())]
    except Exception:  # noqa: BLE001 - collection must not depend on a toolchain
        return []
    return [None] + [n for n in names if n.startswith(prefix)
                     and not any(e in n for e in exclude)]


class _forced:
    def __init__(self, variant):
        self.variant = variant

    def __enter__(self):
        if self.variant is not None:
            fx.mslkb_force_variant(fx.variant_index(self.variant))

    def __exit__(self, *exc):
        if self.variant is not None:
            fx.mslkb_force_variant(-1)


def _scales(n, g, lo=0.01, span=2.0):
    return (torch.rand(n, generator=g) * span + lo).numpy().astype(np.float32)


def _cuda(*xs):
    return [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in xs]


def _poisoned(shape, poison=0x5A5A):
    return torch.full(shape, poison, dtype=torch.int16, device="cuda").view(torch.bfloat16)


# ---------------------------------------------------------------------------------------
# 1024 groups


def _counts(g, G, hi, zero_frac=0.3):
    m = torch.randint(1, hi + 1, (G,), generator=g).numpy().astype(np.int64)
    m[torch.rand(G, generator=g).numpy() < zero_frac] = 0
    return m


def _stacked_cases():
    # K = 256: TMA loads (every variant); K = 200 (K % 16 = 8): the cp.async loader, which
    # only the cp.async variants and the planner serve
    names = _names("stacked", exclude=("blockscale",))
    return ([(v, 256) for v in names] +
            [(v, 200) for v in names if v is None or "cpasync" in v])


@pytest.mark.parametrize("variant,K", _stacked_cases())
def test_max_groups_stacked(orc, variant, K):
    g = torch.Generator().manual_seed(1024 + K)
    G, N = G_MAX, 136
    m = _counts(g, G, 4)
    m[-1] = 9                       # the last group runs past total_M: clamped
    rows = int(m.sum()) - 4
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa, sb = _scales(rows, g), _scales(G * N, g).reshape(G, N)
    tA, tB, tsa, tsb, tm = _cuda(A, B, sa, sb, m)
    out = _poisoned((rows, N))
    with _forced(variant):
        fx.f8f8bf16_rowwise_grouped_stacked(tA, tB, tsa, tsb, tm, out=out)
    torch.cuda.synchronize()
    assert fx.device_status() == fx.MSLKB_DEV_MSIZES_CLAMPED
    ref, clamped = orc.stacked(A, B, sa, sb, m, total_M=rows)
    ab, _ = orc.stacked(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), m, total_M=rows)
    assert clamped
    compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"G=1024 stacked {variant} K={K}")


@pytest.mark.parametrize("variant", _names("dynamic", exclude=("blockscale",)))
def test_max_groups_dynamic_and_batched(orc, variant):
    g = torch.Generator().manual_seed(7)
    G, E, N, K = G_MAX, 5, 136, 256
    zsi = torch.randint(-2, E + 3, (G,), generator=g).numpy().astype(np.int64)
    A = random_codes((G * E, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa, sb = _scales(G * E, g), _scales(G * N, g).reshape(G, N)
    tA, tB, tsa, tsb, tz = _cuda(A, B, sa, sb, zsi)
    out = _poisoned((G * E, N))
    with _forced(variant):
        fx.f8f8bf16_rowwise_grouped_dynamic(tA, tB, tsa, tsb, tz, out=out)
    torch.cuda.synchronize()
    ref = orc.dynamic(A, B, sa, sb, zsi, E)
    ab = orc.dynamic(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), zsi, E)
    compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"G=1024 dynamic {variant}")
    out = _poisoned((G, E, N))
    with _forced(variant):
        fx.f8f8bf16_rowwise_grouped_batched(tA.view(G, E, K), tB, tsa.view(G, E), tsb, out=out)
    torch.cuda.synchronize()
    ref = orc.batched(A, B, sa, sb)
    ab = orc.batched(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb))
    compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"G=1024 batched {variant}")
    assert fx.device_status() == 0


def test_max_groups_offsets(orc):
    g = torch.Generator().manual_seed(8)
    G, N, K = G_MAX, 136, 256
    m = _counts(g, G, 4)
    rows = int(m.sum()) + 3
    incl = np.cumsum(m).astype(np.int32)
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa, sb = _scales(rows, g), _scales(G * N, g).reshape(G, N)
    tA, tB, tsa, tsb, to = _cuda(A, B, sa, sb, incl)
    out = _poisoned((rows, N))
    fx.f8f8bf16_rowwise_grouped_offsets(tA, tB, tsa, tsb, to, out=out)
    torch.cuda.synchronize()
    poison = np.full((rows, N), 0x5A5A, np.uint16)
    ref, _ = orc.offsets(A, B, sa, sb, incl, total_M=rows, out=poison)
    ab, _ = orc.offsets(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), incl, total_M=rows)
    got = bits_of(out).reshape(rows, N)
    owned = int(m.sum())
    assert np.all(got[owned:] == 0x5A5A), "rows past the last group written"
    compare(got[:owned].ravel(), ref[:owned].ravel(), ab[:owned].ravel(), "G=1024 offsets")
    assert fx.device_status() == 0


@pytest.mark.parametrize("variant", _names("ragn_"))
def test_max_groups_ragged_n(orc, variant):
    g = torch.Generator().manual_seed(9)
    G, M, K = G_MAX, 40, 256
    cols = torch.randint(0, 20, (G,), generator=g).numpy()
    total_N = (int(cols.sum()) + 15) // 8 * 8     # a row of the output: whole 16 bytes
    off = np.cumsum(cols).astype(np.int32)
    A = random_codes((G, M, K), g).numpy()
    B = random_codes((total_N, K), g).numpy()
    sa, sb = _scales(G * M, g).reshape(G, M), _scales(total_N, g)
    tA, tB, tsa, tsb, to = _cuda(A, B, sa, sb, off)
    out = _poisoned((M, total_N))
    with _forced(variant):
        fx.f8f8bf16_rowwise_grouped_n_offsets(tA, tB, tsa, tsb, to, out=out)
    torch.cuda.synchronize()
    ref, _ = orc.n_offsets(A, B, sa, sb, off, out=np.full((M, total_N), 0x5A5A, np.uint16))
    ab, _ = orc.n_offsets(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), off)
    got = bits_of(out).reshape(M, total_N)
    owned = int(off[-1])
    assert np.all(got[:, owned:] == 0x5A5A), "columns past the last group written"
    compare(got[:, :owned].ravel(), ref[:, :owned].ravel(), ab[:, :owned].ravel(),
            f"G=1024 ragged N {variant}")
    assert fx.device_status() == 0


@pytest.mark.parametrize("variant", _names("ragk_"))
def test_max_groups_ragged_k(orc, variant):
    g = torch.Generator().manual_seed(10)
    G, M, N = G_MAX, 40, 136
    ks = 16 * torch.randint(0, 5, (G,), generator=g).numpy()
    total_K = int(ks.sum()) + 16
    off = np.cumsum(ks).astype(np.int32)
    A = random_codes((M, total_K), g).numpy()
    B = random_codes((N, total_K), g).numpy()
    sa, sb = _scales(G * M, g).reshape(G, M), _scales(G * N, g).reshape(G, N)
    tA, tB, tsa, tsb, to = _cuda(A, B, sa, sb, off)
    out = _poisoned((G, M, N))
    with _forced(variant):
        fx.f8f8bf16_rowwise_grouped_k_offsets(tA, tB, tsa, tsb, to, out=out)
    torch.cuda.synchronize()
    ref, _ = orc.k_offsets(A, B, sa, sb, off)
    ab, _ = orc.k_offsets(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), off)
    compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"G=1024 ragged K {variant}")
    assert fx.device_status() == 0


def _block_scales(g, rows, G, N, K):
    nkb, nnb = K // 128, N // 128
    return (_scales(rows * nkb, g).reshape(rows, nkb), _scales(G * nnb * nkb, g).reshape(G, nnb, nkb))


@pytest.mark.parametrize("variant", _names("blockscale_"))
def test_max_groups_block_scaled_stacked(orc, variant):
    g = torch.Generator().manual_seed(11)
    G, N, K = G_MAX, 128, 256
    m = _counts(g, G, 3)
    rows = int(m.sum()) + 2
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa, sb = _block_scales(g, rows, G, N, K)
    tA, tB, tsa, tsb, tm = _cuda(A, B, sa, sb, m)
    out = _poisoned((rows, N))
    with _forced(variant):
        fx.f8f8bf16_groupwise_grouped_stacked(tA, tB, tsa, tsb, tm, out=out)
    torch.cuda.synchronize()
    ref, _ = orc.blockwise_stacked(A, B, sa, sb, m, total_M=rows)
    ab, _ = orc.blockwise_stacked(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), m,
                                  total_M=rows)
    got = bits_of(out).reshape(rows, N)
    owned = int(m.sum())
    assert np.all(got[owned:] == 0x5A5A), "rows past the last group written"
    compare(got[:owned].ravel(), ref[:owned].ravel(), ab[:owned].ravel(),
            f"G=1024 block-scaled stacked {variant}")
    assert fx.device_status() == 0


@pytest.mark.parametrize("variant", _names("dynamic_blockscale_"))
def test_max_groups_block_scaled_dynamic(orc, variant):
    g = torch.Generator().manual_seed(12)
    G, E, N, K = G_MAX, 4, 128, 256
    zsi = torch.randint(-1, E + 2, (G,), generator=g).numpy().astype(np.int64)
    A = random_codes((G * E, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa, sb = _block_scales(g, G * E, G, N, K)
    tA, tB, tsa, tsb, tz = _cuda(A, B, sa, sb, zsi)
    out = _poisoned((G * E, N))
    with _forced(variant):
        fx.f8f8bf16_groupwise_grouped_dynamic(tA, tB, tsa, tsb, tz, out=out)
    torch.cuda.synchronize()
    ref = orc.blockwise_dynamic(A, B, sa, sb, zsi, E)
    ab = orc.blockwise_dynamic(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), zsi, E)
    compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"G=1024 block-scaled dynamic {variant}")
    assert fx.device_status() == 0


# ---------------------------------------------------------------------------------------
# more than 2^31 elements


def _codes_gpu(shape, seed):
    """Uniformly random non-NaN E4M3 codes generated on the GPU in slices (a whole
    int32 intermediate of a 2 GB operand would take 8 GB)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    flat = out.view(-1)
    step = 1 << 28
    for s in range(0, flat.numel(), step):
        n = min(step, flat.numel() - s)
        flat[s:s + n] = random_codes((n,), g, device="cuda")
    return out


def _gpu_scales(n, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.rand(n, generator=g, device="cuda") * 2 + 0.01


def _host(*ts):
    return [t.cpu().numpy() for t in ts]


def _past_2_31(rows, *per_row_elems):
    """Rows around the first whose element offset passes 2^31 in each operand."""
    r = []
    for e in per_row_elems:
        first = -(-TWO31 // e)
        r += [first - 1, first, first + 1]
    return [x for x in r if 0 <= x < rows]


def _fill_left(out, what):
    left = int((out.view(torch.int16) == 0x7E7E).sum().item())
    assert left == 0, f"{what}: {left} elements still hold the fill pattern"


def _check_rows(got_t, rows, ref, ab, what):
    got = bits_of(got_t[torch.from_numpy(rows).cuda()]).reshape(ref.shape)
    compare(got.ravel(), ref.ravel(), ab.ravel(), what)


def _sample(rng, bounds, extra):
    """First and last rows of each [lo, hi) range, two random rows of it, and `extra`."""
    rows = []
    for lo, hi in bounds:
        if hi > lo:
            rows += [lo, hi - 1] + list(rng.integers(lo, hi, size=2))
    return np.unique(np.array(rows + list(extra), dtype=np.int64))


@pytest.mark.parametrize("K", [8192, 8200])   # TMA; the cp.async loader (8-byte copies)
def test_over_2_31_stacked(orc, K):
    G, N = 3, 8192
    m = np.array([100000, 0, 170000] if K == 8192 else [131000, 0, 131200], np.int64)
    rows = int(m.sum())
    assert rows * K > TWO31 and rows * N > TWO31
    tA = _codes_gpu((rows, K), 1)
    tB = _codes_gpu((G, N, K), 2)
    tsa, tsb = _gpu_scales(rows, 3), _gpu_scales(G * N, 4).view(G, N)
    out = torch.full((rows, N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fx.f8f8bf16_rowwise_grouped_stacked(tA, tB, tsa, tsb, torch.from_numpy(m).cuda(), out=out)
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    _fill_left(out, f"stacked K={K}")
    sample = _sample(np.random.default_rng(K), [(0, 100000 if K == 8192 else 131000),
                                                (int(m[0]), rows)], _past_2_31(rows, K, N))
    A, B, sa, sb = _host(tA, tB, tsa, tsb)
    ref = orc.stacked_rows(A, B, sa, sb, m, sample)
    ab = orc.stacked_rows(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), m, sample)
    _check_rows(out, sample, ref, ab, f"stacked over 2^31 K={K}")
    del tA, tB, out, A, B
    torch.cuda.empty_cache()


def test_over_2_31_dynamic(orc):
    G, E, N, K = 4, 67000, 8192, 8192
    zsi = np.array([E, 0, 12345, E - 1], np.int64)
    assert G * E * K > TWO31 and G * E * N > TWO31
    tA = _codes_gpu((G * E, K), 5)
    tB = _codes_gpu((G, N, K), 6)
    tsa, tsb = _gpu_scales(G * E, 7), _gpu_scales(G * N, 8).view(G, N)
    out = torch.full((G * E, N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fx.f8f8bf16_rowwise_grouped_dynamic(tA, tB, tsa, tsb, torch.from_numpy(zsi).cuda(), out=out)
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    _fill_left(out, "dynamic")
    for gi in range(G):   # padding rows: +0.0 exactly
        pad = out[gi * E + int(zsi[gi]):(gi + 1) * E].view(torch.int16)
        assert int((pad != 0).sum().item()) == 0, f"group {gi}: a padding row is not +0.0"
    sample = _sample(np.random.default_rng(1), [(g * E, g * E + int(zsi[g])) for g in range(G)],
                     _past_2_31(G * E, K, N))
    A, B, sa, sb = _host(tA, tB, tsa, tsb)
    ref = orc.dynamic_rows(A, B, sa, sb, zsi, E, sample)
    ab = orc.dynamic_rows(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), zsi, E, sample)
    _check_rows(out, sample, ref, ab, "dynamic over 2^31")
    del tA, tB, out, A, B
    torch.cuda.empty_cache()


def test_over_2_31_block_scaled_stacked(orc):
    G, N, K = 2, 8192, 8192
    m = np.array([150000, 120000], np.int64)
    rows = int(m.sum())
    nkb, nnb = K // 128, N // 128
    tA = _codes_gpu((rows, K), 9)
    tB = _codes_gpu((G, N, K), 10)
    tsa = _gpu_scales(rows * nkb, 11).view(rows, nkb)
    tsb = _gpu_scales(G * nnb * nkb, 12).view(G, nnb, nkb)
    out = torch.full((rows, N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fx.f8f8bf16_groupwise_grouped_stacked(tA, tB, tsa, tsb, torch.from_numpy(m).cuda(), out=out)
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    _fill_left(out, "block-scaled stacked")
    sample = _sample(np.random.default_rng(2), [(0, 150000), (150000, rows)],
                     _past_2_31(rows, K, N))
    A, B, sa, sb = _host(tA, tB, tsa, tsb)
    ref, _ = orc.blockwise_stacked(A, B, sa, sb, m, total_M=rows, rows=sample)
    ab, _ = orc.blockwise_stacked(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), m,
                                  total_M=rows, rows=sample)
    _check_rows(out, sample, ref, ab, "block-scaled stacked over 2^31")
    del tA, tB, out, A, B
    torch.cuda.empty_cache()


def test_over_2_31_weights_decode(orc):
    # one row against a single weight matrix of more than 2^31 elements (the decode plans:
    # swap-AB tiles, the weight prefetch, split tiles); N not a multiple of the tile
    G, N, K = 1, 262160, 8192
    assert N * K > TWO31
    tA = _codes_gpu((1, K), 13)
    tB = _codes_gpu((G, N, K), 14)
    tsa, tsb = _gpu_scales(1, 15), _gpu_scales(G * N, 16).view(G, N)
    out = torch.full((1, N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    m = torch.tensor([1], dtype=torch.int64, device="cuda")
    fx.f8f8bf16_rowwise_grouped_stacked(tA, tB, tsa, tsb, m, out=out)
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    _fill_left(out, "decode")
    # the whole output row, against the oracle on column slices of B (each column of the
    # output depends on its own weight row only)
    A, sa = _host(tA, tsa)
    got = bits_of(out).reshape(N)
    for c0 in (0, N // 2 - 4096, N - 8192):
        cols = slice(c0, c0 + 8192)
        B = tB[:, cols].cpu().numpy()
        sb = tsb[:, cols].cpu().numpy()
        ref, _ = orc.stacked(A, B, sa, sb, np.array([1], np.int64))
        ab, _ = orc.stacked(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb),
                            np.array([1], np.int64))
        compare(got[cols], ref.ravel(), ab.ravel(), f"decode over 2^31 columns {c0}..")
    del tA, tB, out
    torch.cuda.empty_cache()


def test_over_2_31_ragged_k(orc):
    G, M, N = 4, 4096, 4096
    off = np.array([131072, 262144, 262144, 532480], np.int32)   # one empty slice
    total_K = int(off[-1])
    assert M * total_K > TWO31 and N * total_K > TWO31
    tA = _codes_gpu((M, total_K), 17)
    tB = _codes_gpu((N, total_K), 18)
    tsa, tsb = _gpu_scales(G * M, 19).view(G, M), _gpu_scales(G * N, 20).view(G, N)
    out = torch.full((G, M, N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fx.f8f8bf16_rowwise_grouped_k_offsets(tA, tB, tsa, tsb, torch.from_numpy(off).cuda(), out=out)
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    _fill_left(out, "ragged K")
    # rows whose A row starts past 2^31 elements, in every slab
    first = -(-TWO31 // total_K)
    sample = np.array(sorted({g * M + r for g in range(G) for r in (0, first - 1, first, M - 1)}),
                      np.int64)
    A, B, sa, sb = _host(tA, tB, tsa, tsb)
    ref, _ = orc.k_offsets(A, B, sa, sb, off, rows=sample)
    ab, _ = orc.k_offsets(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), off, rows=sample)
    _check_rows(out.view(G * M, N), sample, ref, ab, "ragged K over 2^31")
    del tA, tB, out, A, B
    torch.cuda.empty_cache()


def test_over_2_31_ragged_n(orc):
    G, M, K = 2, 131072, 1024
    off = np.array([8200, 16400], np.int32)
    total_N = int(off[-1])
    assert M * total_N > TWO31
    tA = _codes_gpu((G, M, K), 21)
    tB = _codes_gpu((total_N, K), 22)
    tsa, tsb = _gpu_scales(G * M, 23).view(G, M), _gpu_scales(total_N, 24)
    out = torch.full((M, total_N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fx.f8f8bf16_rowwise_grouped_n_offsets(tA, tB, tsa, tsb, torch.from_numpy(off).cuda(), out=out)
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    _fill_left(out, "ragged N")
    sample = _sample(np.random.default_rng(3), [(0, M)], _past_2_31(M, total_N))
    A, B, sa, sb = _host(tA, tB, tsa, tsb)
    ref, _ = orc.n_offsets(A, B, sa, sb, off, rows=sample)
    ab, _ = orc.n_offsets(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), off, rows=sample)
    _check_rows(out, sample, ref, ab, "ragged N over 2^31")
    del tA, tB, out, A, B
    torch.cuda.empty_cache()
