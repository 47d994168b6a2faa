"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element,
on seeded inputs that span several tiles, ragged tails and the layouts' edge cases."""
import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import make_inputs, random_codes, workloads
from parity_util import Problem, bits_of, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fxbuild.build()
    fx.lib()
    fx.device_status()  # start from a clear status word


@pytest.fixture(scope="module")
def orc():
    return oracle.load(0)


def _rand_problem(layout, G, N, K, meta, E=0, seed=0, nan=False, total_extra=0):
    g = torch.Generator().manual_seed(seed)
    if layout == "stacked":
        rows = int(np.clip(np.asarray(meta), 0, None).sum()) + total_extra
    else:
        rows = G * E
    A = random_codes((rows, K), g, allow_nan=nan).numpy()
    B = random_codes((G, N, K), g, allow_nan=nan).numpy()
    sa = (torch.rand(rows, generator=g) * 2 + 0.01).numpy().astype(np.float32)
    sb = (torch.rand(G * N, generator=g) * 2 + 0.01).numpy().astype(np.float32).reshape(G, N)
    return Problem.from_numpy(layout, A, B, sa, sb, meta, expected_m=E)


def _check_full(prob, orc, out=None, variant=None, poison_value=None, what=""):
    """Run the CUDA path, compare every owned element, and check that rows the layout
    does not own kept their previous contents."""
    rows, N = prob.rows, prob.N
    if out is None and poison_value is not None:
        out = torch.full((rows, N), 0, dtype=torch.int16, device="cuda")
        out.fill_(poison_value)
        out = out.view(torch.bfloat16)
    res = prob.run_gpu(out=out, variant=variant)
    torch.cuda.synchronize()
    gb = bits_of(res).reshape(rows, N)
    poison = None
    if poison_value is not None:
        poison = np.full((rows, N), poison_value & 0xFFFF, np.uint16)
    ref, ab = prob.oracle_full(orc, poison=poison)
    owned = prob.owned_rows_mask()
    st = compare(gb[owned].ravel(), ref[owned].ravel(), ab[owned].ravel(), what)
    if poison_value is not None:
        assert np.all(gb[~owned] == (poison_value & 0xFFFF)), f"{what}: unowned rows written"
    return gb, st


# ---------------------------------------------------------------------------------------
# the two small configurations, in full
# ---------------------------------------------------------------------------------------
def test_config0_stacked(orc):
    wl = workloads()["c0_stacked_small"]
    prob = Problem.from_inputs(wl, {k: v.cuda() for k, v in make_inputs(wl, "cpu").items()})
    _, st = _check_full(prob, orc, poison_value=0x7E7E, what="config0")
    assert st["elements"] == 64 * 256
    assert fx.device_status() == 0


def test_config1_dynamic_with_poisoned_padding(orc):
    wl = workloads()["c1_dynamic_tails"]
    inp = {k: v.cuda() for k, v in make_inputs(wl, "cpu").items()}
    prob = Problem.from_inputs(wl, inp)
    gb, st = _check_full(prob, orc, what="config1")
    E, G = wl.expected_m, wl.G
    zsi = list(wl.meta)
    for g in range(G):
        assert np.all(gb.reshape(G, E, -1)[g, zsi[g]:] == 0), f"padding of slab {g} not +0.0"
    # poison the padding rows of A (NaN codes) and their scales (NaN): bit-identical output
    A2 = inp["A"].clone()
    sa2 = inp["scale_a"].clone()
    for g in range(G):
        A2[g * E + zsi[g]:(g + 1) * E] = 0x7F
        sa2[g * E + zsi[g]:(g + 1) * E] = float("nan")
    prob2 = Problem(wl.layout, A2, inp["B"], sa2, inp["scale_b"], inp["meta"], E)
    gb2 = bits_of(prob2.run_gpu()).reshape(G * E, -1)
    assert np.array_equal(gb, gb2), "padding rows of A leaked into the output"


# ---------------------------------------------------------------------------------------
# every kernel variant on ragged shapes: several tiles, K and N tails, empty groups,
# rows past the last group, tiles that overhang into the next group
# ---------------------------------------------------------------------------------------
def _variants(prefix):
    """Variant names from the library's own table (empty if it cannot be built here;
    the tests that use it then fail on a GPU machine rather than at collection)."""
    try:
        fxbuild.build()
        return [fx.variant_name(i) for i in range(fx.mslkb_num_variants())
                if fx.variant_name(i).startswith(prefix)
                and "blockscale" not in fx.variant_name(i)]   # rowwise variants only
    except Exception:  # noqa: BLE001 - collection must not depend on a toolchain
        return []


def test_every_variant_fits_one_sm():
    for i in range(fx.mslkb_num_variants()):
        blocks, regs = fx.mslkb_variant_resources(i)
        assert blocks >= 1, f"{fx.variant_name(i)}: {blocks} CTAs per SM, {regs} registers"


@pytest.mark.parametrize("variant", _variants("stacked"))
def test_stacked_variant_ragged(orc, variant):
    meta = [130, 0, 1, 257, 64, 0, 17]
    prob = _rand_problem("stacked", 7, 392, 688, meta, seed=1, total_extra=9)
    _check_full(prob, orc, variant=variant, poison_value=0x5A5A, what=variant)


@pytest.mark.parametrize("variant", _variants("dynamic"))
def test_dynamic_variant_ragged(orc, variant):
    meta = [0, 130, 200, 7, -4, 999]
    prob = _rand_problem("dynamic", 6, 392, 688, meta, E=200, seed=2)
    gb, _ = _check_full(prob, orc, variant=variant, what=variant)
    v = np.clip(meta, 0, 200)
    for g in range(6):
        assert np.all(gb[g * 200 + v[g]:(g + 1) * 200] == 0)


@pytest.mark.parametrize("layout", ["stacked", "dynamic"])
def test_pair_tiles_many_waves(orc, layout):
    # CTA pairs (256 x 256 output tiles from one cta_group::2 MMA): more tiles than pairs
    # fit on the GPU, so each pair runs several tiles and reuses its TMEM accumulators;
    # groups end inside the leader's rows, inside the peer's rows, or leave the peer none
    if layout == "stacked":
        meta = [520, 3, 0, 700, 256, 129, 511, 520]
        prob = _rand_problem("stacked", 8, 1024, 512, meta, seed=11, total_extra=5)
    else:
        meta = [520, 3, 0, 600, 256, 129, 511, 520]
        prob = _rand_problem("dynamic", 8, 1024, 512, meta, E=600, seed=12)
    v = f"{layout}_pair256x256_tma"
    for kpc in (8, 1):   # one chunk per tile; a chunk per K block
        fx.mslkb_set_accumulation_chunk(kpc)
        try:
            _check_full(prob, orc, variant=v, poison_value=0x5A5A if layout == "stacked" else None,
                        what=f"{v} chunk {kpc}")
        finally:
            fx.mslkb_set_accumulation_chunk(8)
    assert fx.device_status() == 0


@pytest.mark.parametrize("K", [1024, 0])
@pytest.mark.parametrize("layout", ["stacked", "dynamic"])
def test_pair_transposed_remainders(orc, layout, K):
    """A group's last <= 128 rows on CTA pairs run as a transposed tile: the weights as the
    M = 256 operand, the rows, rounded up to 16, as N with half of them in each CTA.
    Remainders of 1 to 128 rows (N = 16 ... 128; shares of 8 to 64 rows per CTA), 129 (a
    whole tile), after zero or one whole tile of the group; N = 520, so that the last
    column tile's second CTA lies wholly past N; one chunk per tile (K = 1024: eight K
    blocks, the unrolled MMA path) and one per K block; K = 0 writes +0.0 to every owned
    row."""
    rems = [1, 15, 16, 17, 31, 48, 64, 65, 96, 112, 113, 127, 128, 129]
    meta = [256 * (i % 2) + r for i, r in enumerate(rems)]
    if layout == "stacked":
        prob = _rand_problem("stacked", len(meta), 520, K, meta, seed=31 + K, total_extra=3)
    else:
        prob = _rand_problem("dynamic", len(meta), 520, K, meta, E=400, seed=32 + K)
    v = f"{layout}_pair256x256_tma"
    for kpc in (8, 1):
        fx.mslkb_set_accumulation_chunk(kpc)
        try:
            gb, _ = _check_full(prob, orc, variant=v,
                                poison_value=0x5A5A if layout == "stacked" else None,
                                what=f"{v} K {K} chunk {kpc}")
        finally:
            fx.mslkb_set_accumulation_chunk(8)
        if K == 0:
            assert np.all(gb[prob.owned_rows_mask()] == 0)
    assert fx.device_status() == 0


@pytest.mark.parametrize("tile", ["tile128x128", "swap_w128xa16"])
@pytest.mark.parametrize("layout", ["stacked", "dynamic"])
def test_cpasync_bit_identical_to_tma(orc, tile, layout):
    """The two loaders fill the same swizzled tiles, so the MMA sequence and the output
    are the same bit for bit."""
    if layout == "stacked":
        prob = _rand_problem("stacked", 4, 264, 1024 + 48, [40, 200, 0, 3], seed=3)
    else:
        prob = _rand_problem("dynamic", 3, 264, 1024 + 48, [40, 77, 0], E=96, seed=3)
    a = bits_of(prob.run_gpu(variant=f"{layout}_{tile}_tma"))
    b = bits_of(prob.run_gpu(variant=f"{layout}_{tile}_cpasync"))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("K", [1000, 1004, 1001, 24, 8, 4, 1, 130])
def test_k_tails_and_copy_widths(orc, K):
    """K not a multiple of 16 (and of 8, 4, 2): the cp.async loader with the widest copy
    K allows, zero fill past K."""
    prob = _rand_problem("stacked", 3, 136, K, [5, 140, 20], seed=K)
    _check_full(prob, orc, poison_value=0x3C3C, what=f"K={K}")
    probd = _rand_problem("dynamic", 2, 136, K, [3, 150], E=160, seed=K + 1)
    _check_full(probd, orc, what=f"dynamic K={K}")


def test_misaligned_A_uses_narrow_copies(orc):
    """A based at an 8-byte (not 16-byte) boundary: served by the 8-byte copy path."""
    K, N, G = 256, 64, 2
    prob = _rand_problem("stacked", G, N, K, [33, 20], seed=5)
    buf = torch.zeros(prob.A.numel() + 16, dtype=torch.uint8, device="cuda")
    buf[8:8 + prob.A.numel()] = prob.A.view(-1)
    out = torch.zeros((prob.rows, N), dtype=torch.bfloat16, device="cuda")
    s = fx.mslkb_f8f8bf16_rowwise_grouped_stacked(
        buf.data_ptr() + 8, prob.B.data_ptr(), prob.sa.data_ptr(), prob.sb.data_ptr(),
        prob.meta.data_ptr(), out.data_ptr(), prob.rows, G, N, K,
        torch.cuda.current_stream().cuda_stream)
    assert s == fx.MSLKB_OK
    torch.cuda.synchronize()
    ref, ab = prob.oracle_full(orc)
    compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), "misaligned A")


def test_k_zero(orc):
    G, N = 3, 64
    A = np.zeros((12, 0), np.uint8)
    B = np.zeros((G, N, 0), np.uint8)
    prob = Problem.from_numpy("stacked", A, B, np.ones(12, np.float32),
                              np.ones((G, N), np.float32), [4, 0, 5])
    gb, _ = _check_full(prob, orc, poison_value=0x1111, what="K=0 stacked")
    assert np.all(gb[:9] == 0) and np.all(gb[9:] == 0x1111)
    probd = Problem.from_numpy("dynamic", np.zeros((G * 8, 0), np.uint8), B,
                               np.ones(G * 8, np.float32), np.ones((G, N), np.float32),
                               [4, 0, 8], expected_m=8)
    out = torch.full((G * 8, N), 0x2222, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    assert np.all(bits_of(probd.run_gpu(out=out)) == 0)


def test_msizes_clamped_and_reported(orc):
    prob = _rand_problem("stacked", 3, 64, 128, [5, -3, 100], seed=7, total_extra=0)
    prob.rows = 20
    prob.A = prob.A[:20].contiguous()
    prob.sa = prob.sa[:20].contiguous()
    prob._host = None
    fx.device_status()
    _check_full(prob, orc, what="clamped m_sizes")
    assert fx.device_status() & fx.MSLKB_DEV_MSIZES_CLAMPED


def test_identity_weights(orc):
    """B = I (N = K): the output reproduces A times its scales (B = I diagnostic)."""
    K = 256
    G = 2
    g = torch.Generator().manual_seed(9)
    A = random_codes((300, K), g).numpy()
    B = np.zeros((G, K, K), np.uint8)
    for i in range(G):
        np.fill_diagonal(B[i], 0x38)
    sa = np.ldexp(np.ones(300), np.arange(300) % 5 - 2).astype(np.float32)
    sb = np.ones((G, K), np.float32)
    prob = Problem.from_numpy("stacked", A, B, sa, sb, [170, 130])
    out = bits_of(prob.run_gpu()).reshape(300, K)
    exp = (torch.from_numpy(A).view(torch.float8_e4m3fn).float() * torch.from_numpy(sa)[:, None])
    exp = exp.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    exp[exp == 0x8000] = 0
    out = out.copy()
    out[out == 0x8000] = 0
    assert np.array_equal(out, exp)


def test_coherent_boundary_groups(orc):
    """Alternate groups hold constant single-signed data, so a tile that reads or writes
    past its group's rows, N end or K end lands orders of magnitude outside tolerance."""
    meta = [129, 1, 127, 0, 255, 33]
    G, N, K = 6, 264, 1040
    rows = sum(meta)
    A = np.zeros((rows, K), np.uint8)
    B = np.zeros((G, N, K), np.uint8)
    off = 0
    for gi, m in enumerate(meta):
        A[off:off + m] = 0x40 if gi % 2 == 0 else 0xB0   # +2 / -0.5
        B[gi] = 0x48 if gi % 2 == 0 else 0x30             # +4 / +0.5
        off += m
    prob = Problem.from_numpy("stacked", A, B, np.ones(rows, np.float32),
                              np.ones((G, N), np.float32), meta)
    for v in _variants("stacked"):
        _check_full(prob, orc, variant=v, what=f"coherent {v}")


def test_layout_agreement_bitwise(orc):
    """The same rows through the stacked and the dynamic layout, same tile shape."""
    meta = [50, 0, 128, 7]
    G, N, K, E = 4, 256, 512, 128
    ps = _rand_problem("stacked", G, N, K, meta, seed=11)
    h = ps.host()
    Ad = np.zeros((G * E, K), np.uint8)
    sad = np.ones(G * E, np.float32)
    off = 0
    for gi, m in enumerate(meta):
        Ad[gi * E:gi * E + m] = h["A"][off:off + m]
        sad[gi * E:gi * E + m] = h["sa"][off:off + m]
        off += m
    pd = Problem.from_numpy("dynamic", Ad, h["B"], sad, h["sb"], meta, expected_m=E)
    # the two layouts plan different grids, so split tiles would be cut differently
    fx.mslkb_set_split_k(0)
    try:
        _layout_agreement(ps, pd, meta, E, N)
    finally:
        fx.mslkb_set_split_k(1)


def _layout_agreement(ps, pd, meta, E, N):
    for tile in ("tile128x128_tma", "tile128x256_tma", "swap_w128xa16_tma"):
        a = bits_of(ps.run_gpu(variant=f"stacked_{tile}")).reshape(-1, N)
        b = bits_of(pd.run_gpu(variant=f"dynamic_{tile}")).reshape(-1, N)
        off = 0
        for gi, m in enumerate(meta):
            assert np.array_equal(a[off:off + m], b[gi * E:gi * E + m]), f"{tile} group {gi}"
            off += m


def test_deterministic_repeat(orc):
    prob = _rand_problem("stacked", 4, 512, 2048, [300, 1, 0, 211], seed=13)
    a = bits_of(prob.run_gpu())
    for _ in range(3):
        assert np.array_equal(a, bits_of(prob.run_gpu()))


def test_output_redzones(orc):
    prob = _rand_problem("stacked", 3, 128, 384, [100, 0, 60], seed=15)
    pad = 4096
    n = prob.rows * prob.N
    big = torch.full((n + 2 * pad,), 0x6B6B, dtype=torch.int16, device="cuda")
    out = big[pad:pad + n].view(torch.bfloat16).view(prob.rows, prob.N)
    for v in _variants("stacked"):
        prob.run_gpu(out=out, variant=v)
        torch.cuda.synchronize()
        hb = big.cpu().numpy()
        assert np.all(hb[:pad] == 0x6B6B) and np.all(hb[pad + n:] == 0x6B6B), v


def test_accumulator_cancellation(orc):
    """K = 16384 where the second half of the products mirrors the first with the opposite
    sign, so the partial sums climb to half of sum|terms| and then cancel to a small
    remainder.  The tolerance is then essentially 1e-6 * sum|terms|: an fp32 accumulator
    that rounds to nearest meets it; a reduced-precision or truncating one misses it."""
    K, N, M = 16384, 128, 24
    g = torch.Generator().manual_seed(17)
    h = K // 2
    a1 = random_codes((M, h), g).numpy() & 0x7F
    b1 = random_codes((1, N, h), g).numpy() & 0x7F
    a = np.concatenate([a1, a1 | 0x80], axis=1)
    b = np.concatenate([b1, b1], axis=2)
    a[:, K - 1] &= 0x7F  # leave a small, nonzero remainder
    prob = Problem.from_numpy("stacked", a, b, np.ones(M, np.float32),
                              np.ones((1, N), np.float32), [M])
    for v in ("stacked_tile128x256_tma", "stacked_tile128x128_tma", "stacked_swap_w128xa32_tma"):
        _check_full(prob, orc, variant=v, what=f"cancellation {v}")


def test_accumulator_cancellation_inside_chunks(orc):
    """The same stress at the scale of one accumulation chunk (the library's current
    chunk length): in every chunk the second half of the products mirrors the first with
    the opposite sign, so each chunk's own partial sums climb and cancel, and the chunk
    totals are ~0 -- the worst case for the tensor core's round-toward-zero adds."""
    half = 64 * fx.mslkb_accumulation_chunk()  # a chunk is 128 K elements per K-block
    K, N, M = 16384, 128, 24
    g = torch.Generator().manual_seed(23)
    a = random_codes((M, K), g).numpy() & 0x7F
    b = random_codes((1, N, K), g).numpy() & 0x7F
    for k0 in range(0, K, 2 * half):
        a[:, k0 + half:k0 + 2 * half] = a[:, k0:k0 + half] | 0x80
        b[:, :, k0 + half:k0 + 2 * half] = b[:, :, k0:k0 + half]
    a[:, K - 1] &= 0x7F
    prob = Problem.from_numpy("stacked", a, b, np.ones(M, np.float32),
                              np.ones((1, N), np.float32), [M])
    for v in ("stacked_tile128x256_tma", "stacked_swap_w128xa32_tma"):
        _check_full(prob, orc, variant=v, what=f"chunk-scale cancellation {v}")


@pytest.mark.parametrize("kpc", [1, 3, 4, 7])
def test_accumulation_chunk_lengths(orc, kpc):
    """Every accepted chunk length stays within tolerance on random data, including a K
    whose last chunk is partial."""
    prob = _rand_problem("stacked", 3, 264, 128 * 13 + 64, [150, 0, 77], seed=21)
    old = fx.mslkb_accumulation_chunk()
    try:
        fx.mslkb_set_accumulation_chunk(kpc)
        for v in ("stacked_tile128x256_tma", "stacked_swap_w128xa32_tma"):
            _check_full(prob, orc, variant=v, what=f"chunk {kpc} {v}")
    finally:
        fx.mslkb_set_accumulation_chunk(old)


@pytest.mark.parametrize("variant,K,G,N,meta,E", [
    # 128x256 tiles, 4 stages: 9 K blocks per tile (a whole 8-block chunk, then one block),
    # so a CTA's k-th tile starts its whole chunk at ring position k mod 4; 31 row tiles x
    # 16 column tiles = 496 tiles give some of the 152 CTAs four tiles
    ("stacked_tile128x256_tma", 128 * 9, 3, 4096, [1280, 1290, 1237], 0),
    # 128x128 tiles, 6 stages: 13 K blocks (13 = 1 mod 6), 49 x 16 = 784 tiles (six per CTA)
    ("stacked_tile128x128_tma", 128 * 13, 3, 2048, [2048, 2100, 1990], 0),
    # CTA pairs, 6 stages, slabs ending in full and half pair tiles: 13 K blocks, 26 x 16 =
    # 416 tiles over 76 pairs (six for some)
    ("dynamic_pair256x256_tma", 128 * 13, 4, 4096, [1600, 1500, 1600, 1345], 1600),
])
def test_unrolled_chunks_at_every_ring_position(orc, variant, K, G, N, meta, E):
    """Whole accumulation chunks are issued from a compile-time unrolled path, one instance
    per ring position; these shapes start whole chunks at every position of the ring."""
    layout = variant.split("_")[0]
    prob = _rand_problem(layout, G, N, K, meta, E=E, seed=31)
    assert fx.mslkb_accumulation_chunk() == 8
    _check_full(prob, orc, variant=variant, what=variant)
    assert fx.device_status() == 0


def test_cuda_graph_replay(orc):
    prob = _rand_problem("stacked", 4, 256, 512, [64, 0, 100, 3], seed=19)
    out = torch.empty((prob.rows, prob.N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        prob.run_gpu(out=out)  # first call on s: one-time set-up outside capture
    s.synchronize()
    eager = bits_of(out)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        prob.run_gpu(out=out)
    out.zero_()
    with torch.cuda.stream(s):
        graph.replay()
    s.synchronize()
    assert np.array_equal(bits_of(out), eager)


@pytest.mark.parametrize("layout", ["stacked", "dynamic"])
def test_pair_tile_claims_across_calls_and_graphs(orc, layout):
    """Stacked CTA-pair plans claim their tiles from a per-stream counter that the last pair
    of each call resets (slab layouts take them in a fixed stride): back-to-back calls, graph
    replays and a capture made before the stream had a counter (fixed stride) all give the
    oracle's result, bit-identical to each other."""
    if layout == "stacked":
        meta = [520, 3, 0, 700, 256, 129, 511, 520]
        prob = _rand_problem("stacked", 8, 4096, 1024 + 128, meta, seed=41, total_extra=5)
    else:
        meta = [520, 3, 0, 600, 256, 129, 511, 520]
        prob = _rand_problem("dynamic", 8, 4096, 1024 + 128, meta, E=600, seed=42)
    # 9 K blocks per tile (an unrolled chunk, then one block); ~220 pair tiles over the pairs
    v = f"{layout}_pair256x256_tma"
    # zeros where the stacked layout owns no rows, so whole outputs compare
    out = torch.zeros((prob.rows, prob.N), dtype=torch.bfloat16, device="cuda")
    fresh = torch.cuda.Stream()
    fresh.wait_stream(torch.cuda.current_stream())
    graph0 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph0, stream=fresh):   # no workspace on this stream yet
        prob.run_gpu(out=out, variant=v)
    with torch.cuda.stream(fresh):
        graph0.replay()
    fresh.synchronize()
    ref_bits, _ = _check_full(prob, orc, out=out.clone(), variant=v, what=f"{v} first call")
    assert np.array_equal(bits_of(out).reshape(prob.rows, prob.N), ref_bits)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            out.zero_()
            prob.run_gpu(out=out, variant=v)
    s.synchronize()
    assert np.array_equal(bits_of(out).reshape(prob.rows, prob.N), ref_bits)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(2):
            prob.run_gpu(out=out, variant=v)
    for _ in range(2):
        out.zero_()
        with torch.cuda.stream(s):
            graph.replay()
        s.synchronize()
        assert np.array_equal(bits_of(out).reshape(prob.rows, prob.N), ref_bits)
    assert fx.device_status() == 0


def test_cuda_graph_on_fresh_stream(orc):
    """Captured on a stream never used before: no workspace can be allocated during
    capture, so the call runs with whole tiles; still within tolerance."""
    prob = _rand_problem("stacked", 4, 256, 1024, [64, 0, 100, 3], seed=20)
    out = torch.zeros((prob.rows, prob.N), dtype=torch.bfloat16, device="cuda")
    fresh = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=fresh):
        prob.run_gpu(out=out)
    with torch.cuda.stream(fresh):
        graph.replay()
    fresh.synchronize()
    ref, ab = prob.oracle_full(orc)
    compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), "graph on a fresh stream")


@pytest.mark.parametrize("shape", ["few_tiles", "one_wave_plus", "many_waves"])
def test_split_tiles(orc, shape):
    """Stream-K: the last waves' tiles are cut along K over all CTAs and finished by the
    last piece.  Split and whole-tile runs both match the oracle; split runs repeat bit
    for bit."""
    if shape == "few_tiles":      # T < #SMs: every tile split into several pieces
        prob = _rand_problem("stacked", 2, 512, 4096, [1, 3], seed=31)
    elif shape == "one_wave_plus":  # #SMs <= T < 2 #SMs
        prob = _rand_problem("stacked", 3, 2048, 1024, [300, 129, 61], seed=32)
    else:                          # T >= 2 #SMs: whole waves, then a split remainder
        prob = _rand_problem("stacked", 4, 4096, 640, [400, 257, 0, 390], seed=33)
    outs = {}
    for split in (2, 0):  # 2: every plan splits, so both tile shapes take the split path
        fx.mslkb_set_split_k(split)
        try:
            for v in ("stacked_tile128x256_tma", "stacked_swap_w128xa16_tma"):
                gb, _ = _check_full(prob, orc, variant=v, what=f"{shape} split={split} {v}")
                outs[(split, v)] = gb
                if split:
                    again = bits_of(prob.run_gpu(variant=v)).reshape(gb.shape)
                    assert np.array_equal(gb, again), f"{shape} {v}: split run not repeatable"
        finally:
            fx.mslkb_set_split_k(1)
    assert fx.device_status() == 0


def test_dynamic_split_tiles(orc):
    prob = _rand_problem("dynamic", 3, 1024, 2048, [5, 0, 77], E=96, seed=34)
    fx.mslkb_set_split_k(2)
    try:
        for v in ("dynamic_tile128x256_tma", "dynamic_swap_w128xa16_tma",
                  "dynamic_tile128x128_cpasync"):
            _check_full(prob, orc, variant=v, what=f"dynamic split {v}")
    finally:
        fx.mslkb_set_split_k(1)


@pytest.mark.parametrize("layout", ["stacked", "dynamic"])
def test_weight_prefetch_is_only_a_hint(orc, layout):
    """Swap-AB plans prefetch weights from a speculative schedule ahead of the dependency
    wait.  The results are bit-identical with the prefetch off, and with the speculation
    reading other metadata -- rows moved to other groups, or counts out of every range --
    so that it prefetches tiles the call never computes."""
    G, N, K = 8, 1024, 4096
    if layout == "stacked":
        prob = _rand_problem("stacked", G, N, K, [0, 3, 0, 9, 1, 0, 16, 2], seed=41)
        fakes = [[31, 0, 0, 0, 0, 0, 0, 0], [2**40, -7, 2**62, 0, -1, 5, 0, 2**33]]
    else:
        prob = _rand_problem("dynamic", G, N, K, [0, 5, 16, 1, 0, 7, 3, 12], E=16, seed=42)
        fakes = [[16, 0, 0, 0, 16, 16, 0, 0], [-3, 2**40, 99, -2**50, 0, 17, 2**31, 1]]
    v = f"{layout}_swap_w128xa16_tma"
    base, _ = _check_full(prob, orc, variant=v, what=f"{layout} prefetch on")
    fx.mslkb_set_weight_prefetch(0)
    try:
        off = bits_of(prob.run_gpu(variant=v)).reshape(base.shape)
    finally:
        fx.mslkb_set_weight_prefetch(-1)
    assert np.array_equal(base, off), f"{layout}: prefetch changed the result"
    for fake in fakes:
        f = torch.tensor(fake, dtype=torch.int64, device="cuda")
        fx.mslkb_test_speculate_from_next_launch(f)
        got = bits_of(prob.run_gpu(variant=v)).reshape(base.shape)
        torch.cuda.synchronize()
        assert np.array_equal(base, got), f"{layout}: speculation from {fake} leaked"
        if layout == "stacked":   # the allocation-free entry point takes the hook too
            out = torch.empty(base.shape, dtype=torch.bfloat16, device="cuda")
            fx.mslkb_test_speculate_from_next_launch(f)
            fx.mslkb_force_variant(fx.variant_index(v))
            try:
                s = fx.mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc(
                    prob.A.data_ptr(), prob.B.data_ptr(), prob.sa.data_ptr(), prob.sb.data_ptr(),
                    prob.meta.data_ptr(), out.data_ptr(), prob.rows, prob.G, prob.N, prob.K,
                    torch.cuda.current_stream().cuda_stream)
            finally:
                fx.mslkb_force_variant(-1)
            assert s == fx.MSLKB_OK, fx.mslkb_status_string(s)
            torch.cuda.synchronize()
            got = bits_of(out).reshape(base.shape)
            assert np.array_equal(base, got), f"allocation-free: speculation from {fake} leaked"
    assert fx.device_status() == 0


@pytest.mark.parametrize("layout", ["stacked", "dynamic"])
def test_many_groups_swap_plan(orc, layout):
    """100 groups of a few rows each (swap-AB plan, split along K): the scheduler's warp
    takes several groups per lane, both in the speculative schedule of the weight prefetch
    and in the real one; empty groups and groups of one row throughout."""
    G, N, K = 100, 256, 1024
    rng = np.random.default_rng(57)
    meta = rng.integers(0, 4, size=G)
    meta[::9] = 0
    if layout == "stacked":
        prob = _rand_problem("stacked", G, N, K, meta.tolist(), seed=58)
    else:
        prob = _rand_problem("dynamic", G, N, K, meta.tolist(), E=4, seed=59)
    _check_full(prob, orc, poison_value=0x5A5A, what=f"{layout}, 100 groups")
    assert fx.device_status() == 0


def test_empty_problems_are_noops():
    dev = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = dev.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    assert fx.mslkb_f8f8bf16_rowwise_grouped_stacked(p, p, p, p, p, p, 0, 4, 64, 64, st) == 0
    assert fx.mslkb_f8f8bf16_rowwise_grouped_stacked(p, p, p, p, p, p, 8, 0, 64, 64, st) == 0
    assert fx.mslkb_f8f8bf16_rowwise_grouped_dynamic(p, p, p, p, p, p, 4, 0, 64, 64, st) == 0
    torch.cuda.synchronize()


def test_no_timeouts_recorded():
    assert fx.device_status() & fx.MSLKB_DEV_TIMEOUT == 0
