"""The checked build, libmslkb_checked.so: the same sources compiled with MSLKB_CHECKED, whose
kernels test every global access -- metadata, scales, TMA coordinates, output stores, the
split-tile workspace -- against the extents of the buffers the call passed, and report an
index outside them in the device status word (MSLKB_DEV_BOUNDS) instead of making the
access.  It stands in for a memory checker, which this GPU pool does not offer.

Every kernel variant of every layout runs through it on problems with ragged ends (groups
ending inside tiles, empty groups, K and N tails, slabs with padding, split tiles, CTA pairs
with tile claims and in a fixed stride, the allocation-free entry point, and the headline
workload at full size), and must match the oracle with nothing reported.  For this module the
Python binding is pointed at the checked library; the product library is restored after it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import make_inputs, workloads
from parity_util import Problem, bits_of, compare

pytestmark = pytest.mark.gpu


_PRODUCT = []   # the product library, while the binding points at the checked one


@pytest.fixture(scope="module", autouse=True)
def checked_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fxbuild.build()
    fx.lib()
    lib = fx.declare(ctypes.CDLL(fxbuild.build(checked=True)))
    saved = fx._lib
    _PRODUCT.append(saved)
    fx._lib = lib
    try:
        fx.device_status()
        yield lib
    finally:
        fx._lib = saved


@pytest.fixture(scope="module")
def orc():
    return oracle.load(0)


def _names(prefix, exclude=()):
    try:
        fxbuild.build()
        names = [fx.variant_name(i) for i in range(fx.mslkb_num_variants())]
    except Exception:  # noqa: BLE001 - collection must not depend on a toolchain
        return []
    return [n for n in names if n.startswith(prefix) and not any(e in n for e in exclude)]


SITES = ["group metadata", "TMA load K coordinate", "TMA load row / column / group coordinate",
         "TMA K coordinate alignment", "scales", "direct output store", "TMA output store",
         "split-tile workspace"]


def _clean(what):
    st = fx.device_status()
    sites = [name for i, name in enumerate(SITES) if st >> (16 + i) & 1]
    assert st & fx.MSLKB_DEV_BOUNDS == 0, f"{what}: an index outside its buffer: {sites}"
    assert st == 0, f"{what}: device status {st:#x}"


def test_the_checked_library_is_the_one_in_use(checked_lib):
    assert fx.lib() is checked_lib
    assert fx.mslkb_version() == 10000


@pytest.mark.parametrize("variant", _names("stacked", exclude=("blockscale",)))
def test_stacked_variants(orc, variant):
    from test_parity import _check_full, _rand_problem
    prob = _rand_problem("stacked", 7, 392, 688, [130, 0, 1, 257, 64, 0, 17], seed=1,
                         total_extra=9)
    _check_full(prob, orc, variant=variant, poison_value=0x5A5A, what=variant)
    _clean(variant)


@pytest.mark.parametrize("variant", _names("dynamic", exclude=("blockscale",)))
def test_dynamic_and_batched_variants(orc, variant):
    from test_parity import _check_full, _rand_problem
    prob = _rand_problem("dynamic", 6, 392, 688, [0, 130, 200, 7, -4, 999], E=200, seed=2)
    _check_full(prob, orc, variant=variant, what=f"{variant} dynamic")
    prob = _rand_problem("batched", 3, 392, 688, [], E=150, seed=3)
    _check_full(prob, orc, variant=variant, what=f"{variant} batched")
    _clean(variant)


def test_offsets_and_k_tails(orc):
    from test_next_layouts import _data, _run_and_check
    from test_parity import _check_full, _rand_problem
    counts = [40, 40, 300, 301, 420]
    A, B, sa, sb = _data(sum(counts) + 5, 5, 264, 512, seed=4)
    po = Problem.from_numpy("offsets", A, B, sa, sb, np.cumsum(counts).astype(np.int32))
    _run_and_check(po, orc, poison=0x5A5A, what="offsets")
    for K in (1000, 1001, 24):  # the cp.async loader at copy widths 8, 1 and 8 bytes
        prob = _rand_problem("stacked", 3, 136, K, [70, 0, 131], seed=5)
        _check_full(prob, orc, what=f"K={K}")
    _clean("offsets and K tails")


@pytest.mark.parametrize("variant", _names("ragn_"))
def test_ragged_n_variants(orc, variant):
    from test_ragged_layouts import _n_offsets_case
    _n_offsets_case(orc, 6, 200, 1032, 400, [0, 3, 300, 517, 1, 203], seed=1, variant=variant)
    _clean(variant)


@pytest.mark.parametrize("variant", _names("ragk_"))
def test_ragged_k_variants(orc, variant):
    from test_ragged_layouts import _k_offsets_case
    _k_offsets_case(orc, 6, 200, 392, 1600, [0, 16, 128, 144, 400, 912], seed=2, variant=variant)
    _clean(variant)


@pytest.mark.parametrize("variant", _names("blockscale_"))
def test_block_scaled_stacked_variants(orc, variant):
    from test_blockscale import _case, _check, _run
    A, B, sa, sb, m, rows = _case(11, 5, [130, 0, 1, 257, 64], 384, 896, extra=5)
    _check(orc, A, B, sa, sb, m, rows, _run(A, B, sa, sb, m, rows, 384, variant), variant)
    _clean(variant)


@pytest.mark.parametrize("variant", _names("dynamic_blockscale_"))
def test_block_scaled_slab_variants(orc, variant):
    from test_blockscale_slabs import _case, _check, _run
    E = 260 if "tile128" in variant else 24
    zsi = [130, 0, 1, E, 5000, -3] if "tile128" in variant else [13, 0, 1, E, 99, -3]
    A, B, sa, sb = _case(21, 6, E, 384, 896, zsi)
    _check(orc, A, B, sa, sb, zsi, E, _run(A, B, sa, sb, zsi, E, variant), variant)
    _clean(variant)


@pytest.mark.parametrize("split", [1, 2])
def test_split_tiles_and_the_allocation_free_call(orc, split):
    from test_parity import _check_full, _rand_problem
    fx.mslkb_set_split_k(split)
    try:
        for meta in ([1, 0, 3, 2, 0, 1, 1, 2], [40, 90, 0, 130, 77, 1, 64, 12]):
            prob = _rand_problem("stacked", 8, 2048, 2048, meta, seed=6)
            _check_full(prob, orc, what=f"split {split} {meta}")
            ref, ab = prob.oracle_full(orc)
            out = torch.empty((prob.rows, prob.N), dtype=torch.bfloat16, device="cuda")
            s = fx.mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc(
                prob.A.data_ptr(), prob.B.data_ptr(), prob.sa.data_ptr(), prob.sb.data_ptr(),
                prob.meta.data_ptr(), out.data_ptr(), prob.rows, prob.G, prob.N, prob.K,
                torch.cuda.current_stream().cuda_stream)
            if s == fx.MSLKB_ERR_TOO_LARGE:   # 128-row tiles split: more than its scratch
                assert split == 2
                continue
            assert s == fx.MSLKB_OK, fx.mslkb_status_string(s)
            torch.cuda.synchronize()
            compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"allocation-free {meta}")
    finally:
        fx.mslkb_set_split_k(1)
    _clean(f"split {split}")


@pytest.mark.parametrize("name", ["c4_llama405b", "c2a_dsv3_gate_up", "c3_llama70b_m1",
                                  "c3_llama70b_m16"])
def test_full_size(orc, name):
    # the planner's kernels on benchmark workloads at full size: CTA pairs claiming their
    # tiles (c4), Zipf-sized groups on 128 x 256 tiles (c2a), split decode tiles (M = 1),
    # decode with two K blocks per weight box (M = 16)
    wl = workloads()[name]
    inp = make_inputs(wl, "cuda")
    prob = Problem.from_inputs(wl, inp)
    out = torch.full((wl.rows, wl.N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    prob.run_gpu(out=out)
    torch.cuda.synchronize()
    _clean(name)
    rows = prob.sample_rows(per_group_random=1, seed=wl.seed, cap=48)
    got = bits_of(out[torch.from_numpy(rows).cuda()]).reshape(rows.size, wl.N)
    ref, ab = prob.oracle_rows(orc, rows)
    compare(got.ravel(), ref.ravel(), ab.ravel(), f"{name} (checked build)")
    del inp, prob, out
    torch.cuda.empty_cache()


LIMITS = [("test_max_groups_stacked", (None, 256)), ("test_max_groups_stacked", (None, 200)),
          ("test_max_groups_dynamic_and_batched", (None,)), ("test_max_groups_offsets", ()),
          ("test_max_groups_ragged_n", (None,)), ("test_max_groups_ragged_k", (None,)),
          ("test_max_groups_block_scaled_stacked", (None,)),
          ("test_max_groups_block_scaled_dynamic", (None,)),
          ("test_over_2_31_stacked", (8192,)), ("test_over_2_31_stacked", (8200,)),
          ("test_over_2_31_dynamic", ()), ("test_over_2_31_weights_decode", ()),
          ("test_over_2_31_ragged_k", ()), ("test_over_2_31_ragged_n", ())]


@pytest.mark.parametrize("name,args", LIMITS, ids=[f"{n}{a}" for n, a in LIMITS])
def test_limits(orc, name, args):
    # 1024 groups on every layout, and operands past 2^31 elements, through the planner's
    # kernels of the checked build (the cases assert a clean status word themselves)
    import test_limits
    fx.device_status()
    getattr(test_limits, name)(orc, *args)
    _clean(name)


@pytest.mark.parametrize("variant", _names("stacked", exclude=("blockscale",)) +
                         _names("dynamic_blockscale_") + _names("blockscale_"))
def test_same_bits_as_the_product_library(checked_lib, variant):
    # the checks change no arithmetic: the same call through both libraries gives the same
    # output bits
    from test_parity import _rand_problem
    outs = []
    for lib in (_PRODUCT[0], checked_lib):
        fx._lib = lib
        try:
            if "blockscale" in variant:
                if variant.startswith("dynamic"):
                    from test_blockscale_slabs import _case, _run
                    zsi = [13, 0, 1, 24, 99, -3]
                    A, B, sa, sb = _case(31, 6, 24, 384, 896, zsi)
                    outs.append(_run(A, B, sa, sb, zsi, 24, variant))
                else:
                    from test_blockscale import _case, _run
                    A, B, sa, sb, m, rows = _case(32, 5, [130, 0, 1, 257, 64], 384, 896, extra=5)
                    outs.append(_run(A, B, sa, sb, m, rows, 384, variant))
            else:
                prob = _rand_problem("stacked", 7, 392, 688, [130, 0, 1, 257, 64, 0, 17], seed=33,
                                     total_extra=9)
                out = torch.full((prob.rows, prob.N), 0x5A5A, dtype=torch.int16,
                                 device="cuda").view(torch.bfloat16)
                prob.run_gpu(out=out, variant=variant)
                torch.cuda.synchronize()
                outs.append(bits_of(out))
        finally:
            fx._lib = checked_lib
    assert np.array_equal(outs[0], outs[1]), f"{variant}: checked and product builds differ"
    _clean(variant)
