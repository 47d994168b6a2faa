"""GPU parity of the block-scaled (groupwise) slab layouts -- dynamic (valid rows at the top of
each group's slab, the rest +0.0) and batched (every slab full) -- against the oracle,
through the C ABI: scale blocks of 128 along K and N, every K block's partial sum scaled on
its way into the fp32 accumulator."""
import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import make_inputs, random_codes, workloads
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
                if fx.variant_name(i).startswith("dynamic_blockscale_")]
    except Exception:  # noqa: BLE001 - collection must not depend on a toolchain
        return []


def _case(seed, G, E, N, K, zsi=None, wide=False, poison_padding=True):
    """Slabs of E rows per group; with zsi, the padding rows of A hold NaN codes and their
    scales NaN (nothing may leak from them)."""
    g = torch.Generator().manual_seed(seed)
    rows = G * E
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    nkb, nnb = K // 128, N // 128
    if wide:   # scales over many binades, so that a scale from the wrong block shows
        sa = np.exp2(torch.randint(-12, 12, (rows, nkb), generator=g).numpy()).astype(np.float32)
        sb = np.exp2(torch.randint(-12, 12, (G, nnb, nkb), generator=g).numpy()).astype(np.float32)
        sa *= (torch.rand((rows, nkb), generator=g).numpy() + 0.5).astype(np.float32)
    else:
        sa = (torch.rand((rows, nkb), generator=g) * 2 + 0.01).numpy().astype(np.float32)
        sb = (torch.rand((G, nnb, nkb), generator=g) * 2 + 0.01).numpy().astype(np.float32)
    if zsi is not None and poison_padding:
        for gi in range(G):
            v = max(0, min(int(zsi[gi]), E))
            A[gi * E + v:(gi + 1) * E] = 0x7F
            sa[gi * E + v:(gi + 1) * E] = np.nan
    return A, B, sa, sb


def _run(A, B, sa, sb, zsi, E, variant=None, poison=0x5A5A):
    G, N, K = B.shape
    tA, tB, tsa, tsb = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (A, B, sa, sb)]
    out = torch.full((G * E, N), poison, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    if variant is not None:
        fx.mslkb_force_variant(fx.variant_index(variant))
    try:
        if zsi is None:
            fx.f8f8bf16_groupwise_grouped_batched(tA.view(G, E, K), tB, tsa, tsb,
                                                  out=out.view(G, E, N))
        else:
            tz = torch.tensor(list(zsi), dtype=torch.int64, device="cuda")
            fx.f8f8bf16_groupwise_grouped_dynamic(tA, tB, tsa, tsb, tz, out=out)
    finally:
        if variant is not None:
            fx.mslkb_force_variant(-1)
    torch.cuda.synchronize()
    return bits_of(out).reshape(G * E, N)


def _check(orc, A, B, sa, sb, zsi, E, got, what):
    """Every slab row: valid rows within tolerance of the oracle, padding rows exactly
    +0.0 (bits 0x0000)."""
    z = None if zsi is None else np.asarray(zsi, np.int64)
    ref = orc.blockwise_dynamic(A, B, sa, sb, z, E)
    # tolerance term from |codes| and |scales|; padding rows hold NaN scales, which the
    # oracle never reads
    ab = orc.blockwise_dynamic(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), z, E)
    if z is not None:
        G = B.shape[0]
        pad = np.concatenate([np.arange(g * E + max(0, min(int(z[g]), E)), (g + 1) * E)
                              for g in range(G)]).astype(np.int64)
        assert np.all(got[pad] == 0x0000), f"{what}: a padding row is not +0.0"
    return compare(got.ravel(), ref.ravel(), ab.ravel(), what)


@pytest.mark.parametrize("variant", _variants())
def test_every_variant_dynamic_and_batched(orc, variant):
    # slabs ending inside tiles, an empty slab, a zero_start_index_M past the slab (clamped)
    # and a negative one (empty), N of 3 scale blocks (a partial 256-wide tile), 7 K blocks
    E = 260 if "tile128" in variant else 24
    zsi = [130, 0, 1, E, 5000, -3] if "tile128" in variant else [13, 0, 1, E, 99, -3]
    A, B, sa, sb = _case(21, 6, E, 384, 896, zsi)
    got = _run(A, B, sa, sb, zsi, E, variant)
    _check(orc, A, B, sa, sb, zsi, E, got, f"{variant} dynamic")
    A, B, sa, sb = _case(22, 3, E, 256, 512)
    got = _run(A, B, sa, sb, None, E, variant)
    _check(orc, A, B, sa, sb, None, E, got, f"{variant} batched")
    assert fx.device_status() == 0


def test_wide_scales_dynamic(orc):
    zsi = [200, 70, 300]
    A, B, sa, sb = _case(23, 3, 300, 512, 1024, zsi, wide=True)
    got = _run(A, B, sa, sb, zsi, 300)
    _check(orc, A, B, sa, sb, zsi, 300, got, "wide scales, dynamic")


@pytest.mark.parametrize("E,zsi", [(16, [1, 0, 3, 16]), (32, [9, 32, 0, 30])])
@pytest.mark.parametrize("split", [1, 0])
def test_decode_slabs(orc, E, zsi, split):
    # few rows per slab: the planner's swap-AB tiles, split along K over every CTA (or not)
    A, B, sa, sb = _case(24, 4, E, 1024, 2048, zsi, wide=True)
    fx.mslkb_set_split_k(split)
    try:
        got = _run(A, B, sa, sb, zsi, E)
    finally:
        fx.mslkb_set_split_k(1)
    _check(orc, A, B, sa, sb, zsi, E, got, f"decode E={E} split={split}")
    assert fx.device_status() == 0


def test_block_scaled_batched_agrees_with_dynamic_full_slabs(orc):
    # the batched call and the dynamic call with every slab full give the same bits
    G, E = 3, 200
    A, B, sa, sb = _case(25, G, E, 256, 640)
    b = _run(A, B, sa, sb, None, E)
    d = _run(A, B, sa, sb, [E] * G, E)
    assert np.array_equal(b, d)
    _check(orc, A, B, sa, sb, None, E, b, "batched")


def test_k_zero_slabs():
    # an empty reduction: every valid row +0.0, and so is every padding row
    for zsi in ([5, 0, 8], None):
        out = torch.full((3 * 8, 128), 1.0, dtype=torch.bfloat16, device="cuda")
        A = torch.zeros((3 * 8, 0), dtype=torch.uint8, device="cuda")
        B = torch.zeros((3, 128, 0), dtype=torch.uint8, device="cuda")
        if zsi is None:
            fx.f8f8bf16_groupwise_grouped_batched(A.view(3, 8, 0), B, torch.ones(0, device="cuda"),
                                                  torch.ones(0, device="cuda"),
                                                  out=out.view(3, 8, 128))
        else:
            fx.f8f8bf16_groupwise_grouped_dynamic(A, B, torch.ones(0, device="cuda"),
                                                  torch.ones(0, device="cuda"),
                                                  torch.tensor(zsi, device="cuda"), out=out)
        torch.cuda.synchronize()
        assert torch.count_nonzero(out.view(torch.int16)).item() == 0
    assert fx.device_status() == 0


@pytest.mark.parametrize("name", ["n7_groupwise_batched_llama70b_m512",
                                  "n8_groupwise_dynamic_dsv3_m256"])
def test_full_size_sampled(orc, name):
    # the benchmark's workloads at full size in the benchmark's plan: sampled slab rows
    # (first, last, last valid, first padding and a random valid row of every slab) in full
    wl = workloads()[name]
    inp = make_inputs(wl, "cuda")
    G, E, N, K = wl.G, wl.expected_m, wl.N, wl.K
    out = torch.full((G * E, N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    st = torch.cuda.current_stream().cuda_stream
    if wl.layout == "groupwise_batched":
        s = fx.mslkb_f8f8bf16_groupwise_grouped_batched(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), out.data_ptr(), G, E, N, K, st)
        zsi = None
    else:
        s = fx.mslkb_f8f8bf16_groupwise_grouped_dynamic(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), G, E, N, K, st)
        zsi = np.asarray(wl.meta, np.int64)
    assert s == fx.MSLKB_OK, fx.mslkb_status_string(s)
    torch.cuda.synchronize()
    rng = np.random.default_rng(wl.seed)
    rows = []
    for g in range(G):
        v = E if zsi is None else max(0, min(int(zsi[g]), E))
        rows += [g * E, g * E + E - 1]
        if v > 0:
            rows += [g * E + v - 1, g * E + int(rng.integers(0, v))]
        if v < E:
            rows += [g * E + v]
    rows = np.unique(np.array(rows, np.int64))
    got = bits_of(out[torch.from_numpy(rows).cuda()]).reshape(rows.size, N)
    h = {k: v.cpu().numpy() for k, v in inp.items()}
    ref = orc.blockwise_dynamic(h["A"], h["B"], h["scale_a"], h["scale_b"], zsi, E, rows=rows)
    ab = orc.blockwise_dynamic(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["scale_a"]),
                               np.abs(h["scale_b"]), zsi, E, rows=rows)
    compare(got.ravel(), ref.ravel(), ab.ravel(), name)
    assert fx.device_status() == 0
    del inp, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("i", range(10))
def test_fuzz_block_scaled_slabs(orc, i):
    rng = np.random.default_rng(7300 + i)
    G = int(rng.integers(1, 9))
    E = int(rng.choice([3, 16, 30, 150, 300]))
    batched = bool(rng.random() < 0.3)
    zsi = None if batched else rng.integers(-2, E + 3, size=G).tolist()
    N = 128 * int(rng.integers(1, 5))
    K = 128 * int(rng.integers(1, 9))
    A, B, sa, sb = _case(7400 + i, G, E, N, K, zsi, wide=bool(rng.random() < 0.5))
    got = _run(A, B, sa, sb, zsi, E)
    _check(orc, A, B, sa, sb, zsi, E, got,
           f"block-scaled slabs #{i}: G={G} E={E} N={N} K={K} zsi={zsi}")
    assert fx.device_status() == 0


@pytest.mark.parametrize("layout", ["dynamic", "batched"])
def test_cuda_graph_replay(orc, layout):
    """The block-scaled slab calls captured in a CUDA graph (after one eager call on the
    stream, which sets up its workspace) and replayed twice, with new inputs copied into
    the captured buffers between the replays."""
    G, E, N, K = 4, 16, 1024, 1024   # decode-sized slabs: swap-AB tiles split along K
    zsi = [3, 16, 0, 9] if layout == "dynamic" else None
    cases = [_case(90 + i, G, E, N, K, zsi) for i in range(2)]
    dev = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in cases[0]]
    tz = None if zsi is None else torch.tensor(zsi, dtype=torch.int64, device="cuda")
    out = torch.empty((G * E, N), dtype=torch.bfloat16, device="cuda")

    def call():
        tA, tB, tsa, tsb = dev
        if tz is None:
            fx.f8f8bf16_groupwise_grouped_batched(tA.view(G, E, K), tB, tsa, tsb,
                                                  out=out.view(G, E, N))
        else:
            fx.f8f8bf16_groupwise_grouped_dynamic(tA, tB, tsa, tsb, tz, out=out)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    for i, (A, B, sa, sb) in enumerate(cases):
        for d, h in zip(dev, (A, B, sa, sb)):
            d.copy_(torch.from_numpy(np.ascontiguousarray(h)))
        with torch.cuda.stream(s):
            graph.replay()
        s.synchronize()
        _check(orc, A, B, sa, sb, zsi, E, bits_of(out).reshape(G * E, N),
               f"{layout} graph replay {i + 1}")
    del graph
    assert fx.device_status() == 0
