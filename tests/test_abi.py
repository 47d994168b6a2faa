"""C-ABI checks that need no GPU: the library builds, loads and exports every symbol
include/*.h declare; argument errors are reported before any CUDA call; the host
planner picks the intended kernel variant for each workload shape."""
import os
import re

import pytest

import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("mslkb.h", "mslkb_tuning.h")]


@pytest.fixture(scope="module")
def L():
    fxbuild.build()
    return fx.lib()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"MSLKB_API\s+[\w\s\*]*?\b(mslkb_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    assert "mslkb_f8f8bf16_rowwise_grouped_stacked" in names
    assert "mslkb_f8f8bf16_rowwise_grouped_dynamic" in names
    assert len(names) >= 10


def test_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} not exported"


def test_exports_nothing_else(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fx.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_functions())


def test_status_strings(L):
    for s in range(7):
        assert fx.mslkb_status_string(s) != "unknown status"
    assert fx.mslkb_status_string(99) == "unknown status"
    assert fx.mslkb_version() == 10000


def _stacked(**kw):
    a = dict(A=16, B=16, scale_a=16, scale_b=16, m_sizes=16, out=256, total_M=4, G=2, N=8, K=16)
    a.update(kw)
    return fx.mslkb_f8f8bf16_rowwise_grouped_stacked(a["A"], a["B"], a["scale_a"], a["scale_b"],
                                                     a["m_sizes"], a["out"], a["total_M"],
                                                     a["G"], a["N"], a["K"], 0)


def _dynamic(**kw):
    a = dict(A=16, B=16, scale_a=16, scale_b=16, zsi=16, out=256, G=2, E=4, N=8, K=16)
    a.update(kw)
    return fx.mslkb_f8f8bf16_rowwise_grouped_dynamic(a["A"], a["B"], a["scale_a"], a["scale_b"],
                                                     a["zsi"], a["out"], a["G"], a["E"], a["N"],
                                                     a["K"], 0)


@pytest.mark.parametrize("call", [_stacked, _dynamic], ids=["stacked", "dynamic"])
def test_argument_errors_before_cuda(L, call):
    # These return before any CUDA call, so they behave the same with or without a GPU.
    assert call(N=12) == fx.MSLKB_ERR_SHAPE          # N not a multiple of 8
    assert call(K=-1) == fx.MSLKB_ERR_SHAPE
    assert call(G=-1) == fx.MSLKB_ERR_SHAPE
    assert call(G=fx.MAX_GROUPS + 1) == fx.MSLKB_ERR_SHAPE
    assert call(N=1 << 33) == fx.MSLKB_ERR_SHAPE     # beyond 32-bit sizes
    assert call(out=0) == fx.MSLKB_ERR_NULL
    assert call(scale_a=0) == fx.MSLKB_ERR_NULL
    assert call(scale_b=0) == fx.MSLKB_ERR_NULL
    assert call(A=0) == fx.MSLKB_ERR_NULL
    assert call(B=0) == fx.MSLKB_ERR_NULL
    assert call(out=264) == fx.MSLKB_ERR_ALIGN       # 8-byte aligned only
    # nothing owned or written: OK without touching the device
    assert call(G=0) == fx.MSLKB_OK
    assert call(N=0) == fx.MSLKB_OK
    assert call(A=0, B=0, K=0, G=0) == fx.MSLKB_OK


def test_argument_errors_layout_specific(L):
    assert _stacked(total_M=-1) == fx.MSLKB_ERR_SHAPE
    assert _stacked(total_M=0) == fx.MSLKB_OK
    assert _stacked(m_sizes=0) == fx.MSLKB_ERR_NULL
    assert _dynamic(E=-1) == fx.MSLKB_ERR_SHAPE
    assert _dynamic(E=0) == fx.MSLKB_OK
    assert _dynamic(zsi=0) == fx.MSLKB_ERR_NULL
    assert _dynamic(G=1024, E=1 << 22) == fx.MSLKB_ERR_SHAPE  # G * E beyond 32 bits
    # K = 0 needs no A or B
    assert _stacked(A=0, B=0, K=0, G=0) == fx.MSLKB_OK


def test_offsets_and_batched_argument_errors(L):
    off = lambda **kw: fx.mslkb_f8f8bf16_rowwise_grouped_offsets(
        *[kw.get(k, d) for k, d in (("A", 16), ("B", 16), ("sa", 16), ("sb", 16), ("o", 16),
                                     ("out", 256), ("M", 4), ("G", 2), ("N", 8), ("K", 16))], 0)
    bat = lambda **kw: fx.mslkb_f8f8bf16_rowwise_grouped_batched(
        *[kw.get(k, d) for k, d in (("A", 16), ("B", 16), ("sa", 16), ("sb", 16),
                                     ("out", 256), ("G", 2), ("M", 4), ("N", 8), ("K", 16))], 0)
    assert off(N=12) == fx.MSLKB_ERR_SHAPE and bat(N=12) == fx.MSLKB_ERR_SHAPE
    assert off(o=0) == fx.MSLKB_ERR_NULL
    assert off(out=264) == fx.MSLKB_ERR_ALIGN and bat(out=264) == fx.MSLKB_ERR_ALIGN
    assert bat(sa=0) == fx.MSLKB_ERR_NULL and bat(M=-1) == fx.MSLKB_ERR_SHAPE
    assert off(M=0) == fx.MSLKB_OK and bat(M=0) == fx.MSLKB_OK and bat(G=0) == fx.MSLKB_OK


def test_ragged_argument_errors(L):
    rn = lambda **kw: fx.mslkb_f8f8bf16_rowwise_grouped_n_offsets(
        *[kw.get(k, d) for k, d in (("A", 256), ("B", 256), ("sa", 16), ("sb", 16), ("o", 16),
                                     ("out", 256), ("G", 2), ("M", 4), ("N", 16), ("K", 32))], 0)
    rk = lambda **kw: fx.mslkb_f8f8bf16_rowwise_grouped_k_offsets(
        *[kw.get(k, d) for k, d in (("A", 256), ("B", 256), ("sa", 16), ("sb", 16), ("o", 16),
                                     ("out", 256), ("G", 2), ("M", 4), ("N", 16), ("K", 32))], 0)
    for call in (rn, rk):
        assert call(N=12) == fx.MSLKB_ERR_SHAPE          # output width not a multiple of 8
        assert call(G=fx.MAX_GROUPS + 1) == fx.MSLKB_ERR_SHAPE
        assert call(M=-1) == fx.MSLKB_ERR_SHAPE
        assert call(o=0) == fx.MSLKB_ERR_NULL and call(sa=0) == fx.MSLKB_ERR_NULL
        assert call(A=0) == fx.MSLKB_ERR_NULL
        assert call(out=264) == fx.MSLKB_ERR_ALIGN
        assert call(K=40) == fx.MSLKB_ERR_ALIGN          # rows of A / B: TMA needs 16-byte steps
        assert call(A=264) == fx.MSLKB_ERR_ALIGN and call(B=264) == fx.MSLKB_ERR_ALIGN
        assert call(M=0) == fx.MSLKB_OK and call(G=0) == fx.MSLKB_OK and call(N=0) == fx.MSLKB_OK
        assert call(A=0, B=0, M=0) == fx.MSLKB_OK


def test_plan_ragged(L):
    # ragged N: tiles over each group's own columns; ragged K: a slab per group; never split
    i = fx.mslkb_plan(2, 1024, 16, 16384, 8192, 152)
    assert fx.variant_name(i.variant) == "ragn_tile128x256_tma" and i.split_k == 0
    assert i.tiles_bound == 8 * (-(-(16384 + 7 * 16) // 256) + 16)
    i = fx.mslkb_plan(2, 16, 16, 4096, 1024, 152)
    assert fx.variant_name(i.variant) == "ragn_swap_w128xa32_tma" and i.split_k == 0
    i = fx.mslkb_plan(3, 4096, 8, 4096, 65536, 152)
    assert fx.variant_name(i.variant) == "ragk_tile128x256_tma" and i.tiles_bound == 8 * 32 * 16
    i = fx.mslkb_plan(3, 128, 2, 256, 1024, 152)
    assert fx.variant_name(i.variant) == "ragk_tile128x128_tma"
    with pytest.raises(fx.MslkbError):
        fx.mslkb_plan(3, 128, 2, 256, 1000, 152)   # K not a multiple of 16: TMA only
    with pytest.raises(fx.MslkbError):
        fx.mslkb_plan(6, 128, 2, 256, 1024, 152)


def test_plan_blockscale_slabs(L):
    """Block-scaled dynamic / batched slabs (layout 5, rows = slab height): swap-AB up to 32
    rows per slab, 128 x 256 tiles when they fill the SMs, else 128 x 128; whole scale
    blocks along K and N, TMA only."""
    i = fx.mslkb_plan(5, 512, 16, 8192, 8192, 152)
    assert fx.variant_name(i.variant) == "dynamic_blockscale_tile128x256_tma"
    i = fx.mslkb_plan(5, 200, 2, 256, 1024, 152)
    assert fx.variant_name(i.variant) == "dynamic_blockscale_tile128x128_tma"
    i = fx.mslkb_plan(5, 16, 8, 4096, 2048, 152)
    assert fx.variant_name(i.variant) == "dynamic_blockscale_swap_w128xa16_tma"
    assert i.split_k == 1
    i = fx.mslkb_plan(5, 32, 8, 4096, 2048, 152)
    assert fx.variant_name(i.variant) == "dynamic_blockscale_swap_w128xa32_tma"
    for bad in ((5, 64, 2, 256, 1000), (5, 64, 2, 200, 1024)):
        with pytest.raises(fx.MslkbError):
            fx.mslkb_plan(*bad, 152)
    with pytest.raises(fx.MslkbError):  # unaligned bases: no cp.async block-scaled kernel
        fx.mslkb_plan(5, 64, 2, 256, 1024, 152, a_align=8)


def _groupwise_dynamic(**kw):
    a = dict(A=16, B=16, scale_a=16, scale_b=16, zsi=16, out=256, G=2, E=4, N=128, K=128)
    a.update(kw)
    return fx.mslkb_f8f8bf16_groupwise_grouped_dynamic(a["A"], a["B"], a["scale_a"],
                                                       a["scale_b"], a["zsi"], a["out"], a["G"],
                                                       a["E"], a["N"], a["K"], 0)


def _groupwise_batched(**kw):
    a = dict(A=16, B=16, scale_a=16, scale_b=16, out=256, G=2, E=4, N=128, K=128)
    a.update(kw)
    return fx.mslkb_f8f8bf16_groupwise_grouped_batched(a["A"], a["B"], a["scale_a"],
                                                       a["scale_b"], a["out"], a["G"], a["E"],
                                                       a["N"], a["K"], 0)


@pytest.mark.parametrize("call", [_groupwise_dynamic, _groupwise_batched],
                         ids=["dynamic", "batched"])
def test_groupwise_slab_argument_errors_before_cuda(L, call):
    assert call(K=192) == fx.MSLKB_ERR_SHAPE          # K not whole scale blocks
    assert call(N=136) == fx.MSLKB_ERR_SHAPE          # N not whole scale blocks
    assert call(E=-1) == fx.MSLKB_ERR_SHAPE
    assert call(G=fx.MAX_GROUPS + 1) == fx.MSLKB_ERR_SHAPE
    assert call(out=0) == fx.MSLKB_ERR_NULL
    assert call(scale_a=0) == fx.MSLKB_ERR_NULL
    assert call(out=264) == fx.MSLKB_ERR_ALIGN        # out not 16-byte aligned
    assert call(G=0) == fx.MSLKB_OK and call(E=0) == fx.MSLKB_OK   # nothing owned


def test_groupwise_argument_errors_and_plan(L):
    gw = lambda **kw: fx.mslkb_f8f8bf16_groupwise_grouped_stacked(
        *[kw.get(k, d) for k, d in (("A", 256), ("B", 256), ("sa", 16), ("sb", 16), ("m", 16),
                                     ("out", 256), ("M", 4), ("G", 2), ("N", 128), ("K", 256))], 0)
    assert gw(K=192) == fx.MSLKB_ERR_SHAPE       # K not whole scale blocks
    assert gw(N=136) == fx.MSLKB_ERR_SHAPE       # N not whole scale blocks
    assert gw(m=0) == fx.MSLKB_ERR_NULL and gw(sb=0) == fx.MSLKB_ERR_NULL
    assert gw(out=264) == fx.MSLKB_ERR_ALIGN
    assert gw(M=0) == fx.MSLKB_OK and gw(G=0) == fx.MSLKB_OK
    i = fx.mslkb_plan(4, 16384, 16, 16384, 16384, 152)
    assert fx.variant_name(i.variant) == "blockscale_tile128x256_tma" and i.split_k == 0
    i = fx.mslkb_plan(4, 512, 4, 256, 512, 152)
    assert fx.variant_name(i.variant) == "blockscale_tile128x128_tma"
    i = fx.mslkb_plan(4, 64, 4, 256, 512, 152)     # 16 rows per group: swap-AB, split along K
    assert fx.variant_name(i.variant) == "blockscale_swap_w128xa16_tma" and i.split_k == 1
    i = fx.mslkb_plan(4, 100, 4, 256, 512, 152)
    assert fx.variant_name(i.variant) == "blockscale_swap_w128xa32_tma"
    with pytest.raises(fx.MslkbError):
        fx.mslkb_plan(4, 64, 4, 256, 520, 152)


def test_accumulation_chunk_setting(L):
    """Only chunk lengths that keep the tolerance (1-8 K blocks) are accepted; a rejected
    value leaves the setting as it was."""
    old = fx.mslkb_accumulation_chunk()
    assert old == 8
    try:
        fx.mslkb_set_accumulation_chunk(1)
        assert fx.mslkb_accumulation_chunk() == 1
        for bad in (0, -1, 9, 16, 1 << 20):
            with pytest.raises(fx.MslkbError):
                fx.mslkb_set_accumulation_chunk(bad)
            assert fx.mslkb_accumulation_chunk() == 1
    finally:
        fx.mslkb_set_accumulation_chunk(old)
    assert fx.mslkb_accumulation_chunk() == 8


def test_hooks_live_in_their_own_header():
    """The process-global tuning and test hooks are declared apart from the entry points."""
    def declared(path):
        return set(re.findall(r"MSLKB_API\s+[\w\s\*]*?\b(mslkb_\w+)\s*\(", open(path).read()))
    main, tuning = declared(HEADERS[0]), declared(HEADERS[1])
    assert not main & tuning
    for name in ("mslkb_force_variant", "mslkb_set_split_k", "mslkb_set_accumulation_chunk",
                 "mslkb_set_weight_prefetch", "mslkb_test_stall_next_launch",
                 "mslkb_test_speculate_from_next_launch"):
        assert name in tuning and name not in main


def test_variant_table(L):
    n = fx.mslkb_num_variants()
    names = [fx.variant_name(i) for i in range(n)]
    assert all(names) and len(set(names)) == n
    assert fx.variant_name(n) is None and fx.variant_name(-1) is None
    for layout in ("stacked", "dynamic"):
        for v in ("tile128x256_tma", "tile128x128_tma", "swap_w128xa16_tma", "tile128x128_cpasync"):
            assert f"{layout}_{v}" in names
    with pytest.raises(fx.MslkbError):
        fx.mslkb_force_variant(n)
    fx.mslkb_force_variant(-1)


GB300_SMS = 152


@pytest.mark.parametrize("name,expect", [
    ("c0_stacked_small", "stacked_swap_w128xa16_tma"),
    ("c1_dynamic_tails", "dynamic_tile128x128_cpasync"),
    ("c2a_dsv3_gate_up", "stacked_tile128x256_tma"),
    ("c2b_dsv3_down", "stacked_tile128x256_tma"),
    ("c3_llama70b_m1", "stacked_swap_w128xa16_tma"),
    ("c3_llama70b_m16", "stacked_swap_w128xa16_tma"),
    ("c3_llama70b_m128", "stacked_swap_w128xa16_tma"),
    ("c3_llama70b_m1024", "stacked_tile128x256_tma"),
    ("c3_llama70b_m8192", "stacked_pair256x256_tma"),
    ("c4_llama405b", "stacked_pair256x256_tma"),
    ("n1_batched_llama70b_m512", "dynamic_pair256x256_tma"),
    ("n2_offsets_llama70b_m8192", "stacked_pair256x256_tma"),
])
def test_plan_per_workload(L, name, expect):
    wl = workloads()[name]
    layout = 1 if wl.slabs else 0   # offsets plan as stacked, batched as dynamic
    rows = wl.expected_m if wl.slabs else wl.rows
    info = fx.mslkb_plan(layout, rows, wl.G, wl.N, wl.K, GB300_SMS)
    assert fx.variant_name(info.variant) == expect
    assert 1 <= info.grid <= GB300_SMS
    assert info.smem_bytes <= 232448
    assert info.threads in (192, 224, 320, 384, 416)


def test_plan_copy_width(L):
    # TMA needs K % 16 == 0 and 16-byte aligned bases; otherwise the copy width follows
    # the largest of 16 / 8 / 4 / 1 that K and both alignments allow
    assert fx.mslkb_plan(0, 512, 4, 256, 512, 152).tma == 1
    i = fx.mslkb_plan(0, 512, 4, 256, 1000, 152)
    assert (i.tma, i.copy_width) == (0, 8)
    i = fx.mslkb_plan(0, 512, 4, 256, 512, 152, a_align=8)
    assert (i.tma, i.copy_width) == (0, 8)
    assert fx.mslkb_plan(0, 512, 4, 256, 1004, 152).copy_width == 4
    assert fx.mslkb_plan(0, 512, 4, 256, 1001, 152).copy_width == 1
    assert fx.mslkb_plan(0, 512, 4, 256, 0, 152).tma == 1


def test_plan_forced_variant(L):
    try:
        fx.mslkb_force_variant(fx.variant_index("dynamic_tile128x128_tma"))
        with pytest.raises(fx.MslkbError):   # wrong layout
            fx.mslkb_plan(0, 512, 4, 256, 512, 152)
        assert fx.mslkb_plan(1, 128, 4, 256, 512, 152).variant == \
            fx.variant_index("dynamic_tile128x128_tma")
        with pytest.raises(fx.MslkbError):   # TMA variant, K not a multiple of 16
            fx.mslkb_plan(1, 128, 4, 256, 1000, 152)
    finally:
        fx.mslkb_force_variant(-1)


def test_plan_pair_variant(L):
    # CTA pairs: 256 x 256 output tiles, two CTAs per tile (an even grid), never split
    try:
        fx.mslkb_force_variant(fx.variant_index("stacked_pair256x256_tma"))
        fx.mslkb_set_split_k(2)
        i = fx.mslkb_plan(0, 16384, 16, 16384, 16384, 152)
        assert (i.tile_m, i.tile_n, i.split_k, i.grid, i.threads) == (256, 256, 0, 152, 384)
        i = fx.mslkb_plan(0, 300, 1, 512, 1024, 152)   # 2 x 2 tiles: 4 pairs
        assert (i.tiles_bound, i.grid) == (4, 8)
        i = fx.mslkb_plan(0, 300, 1, 512, 1024, 7)     # 7 SMs hold 3 pairs
        assert i.grid == 6
        with pytest.raises(fx.MslkbError):             # a stacked kernel for the dynamic layout
            fx.mslkb_plan(1, 128, 4, 256, 512, 152)
        fx.mslkb_force_variant(fx.variant_index("dynamic_pair256x256_tma"))
        i = fx.mslkb_plan(1, 600, 8, 1024, 512, 152)   # 8 slabs x 3 x 4 tiles
        assert (i.tiles_bound, i.grid) == (96, 152)
    finally:
        fx.mslkb_force_variant(-1)
        fx.mslkb_set_split_k(1)


def test_plan_grid_bounds(L):
    # tiles bound for stacked: (total_M + nz * (tile_m - 1)) / tile_m * ceil(N / tile_n)
    try:
        fx.mslkb_set_split_k(0)  # whole tiles: one CTA per tile at most
        i = fx.mslkb_plan(0, 1, 16, 8192, 8192, 152)
        assert i.tiles_bound == 64 and i.grid == 64 and i.split_k == 0
        i = fx.mslkb_plan(1, 128, 8, 1000, 1000, 152)
        assert i.tiles_bound == 8 * 1 * 8 and i.grid == 64
        fx.mslkb_set_split_k(1)  # auto: swap-AB plans split, every SM gets K work
        i = fx.mslkb_plan(0, 1, 16, 8192, 8192, 152)
        assert i.tiles_bound == 64 and i.grid == 152 and i.split_k == 1
        i = fx.mslkb_plan(0, 16384, 64, 16384, 16384, 152)  # 128-row tiles: whole
        assert i.grid == 152 and i.tiles_bound == (16384 + 64 * 127) // 128 * 64
        assert i.split_k == 0 and i.tile_m == 128
        i = fx.mslkb_plan(0, 64, 4, 256, 0, 152)  # K = 0: nothing to split
        assert i.split_k == 0
        fx.mslkb_set_split_k(2)  # every plan
        assert fx.mslkb_plan(0, 16384, 64, 16384, 16384, 152).split_k == 1
        assert fx.mslkb_plan(1, 1024, 16, 16384, 16384, 152).split_k == 0  # pairs: whole
        assert fx.mslkb_plan(0, 512, 2, 4096, 64, 152).grid == 152
        with pytest.raises(fx.MslkbError):
            fx.mslkb_set_split_k(3)
    finally:
        fx.mslkb_set_split_k(1)
