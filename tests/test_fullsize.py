"""GPU parity at the full workload sizes, in the launch configuration the benchmark times
(the host heuristic's variant): every row the oracle computes is compared in full (all
N columns, including the N tail); rows are sampled per group (first, last and random
rows of every non-empty group), since the oracle cannot afford whole outputs here."""
import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import make_inputs, workloads
from parity_util import Problem, bits_of, compare

pytestmark = pytest.mark.gpu

FULL = ["c2a_dsv3_gate_up", "c2b_dsv3_down", "c3_llama70b_m1", "c3_llama70b_m16",
        "c3_llama70b_m128", "c3_llama70b_m1024", "c3_llama70b_m8192", "c4_llama405b",
        "n1_batched_llama70b_m512", "n2_offsets_llama70b_m8192"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fxbuild.build()
    fx.lib()


@pytest.fixture(scope="module")
def orc():
    return oracle.load(0)


def _no_tile_skipped(out, owned, what):
    """Beyond the sampled rows, on the GPU: no owned row still holds the 0x7E7E fill (a tile
    skipped by the scheduler, the claim counter or a split), and nothing is NaN or Inf (the
    inputs hold neither, so a tile written twice with garbage or a lost partial sum would
    show)."""
    owned_t = torch.from_numpy(np.asarray(owned)).cuda()
    o = out[owned_t]
    left = int((o.view(torch.int16) == 0x7E7E).sum().item())
    assert left == 0, f"{what}: {left} owned elements still hold the fill pattern"
    assert bool(torch.isfinite(o).all().item()), f"{what}: NaN or Inf in the output"


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(orc, name):
    wl = workloads()[name]
    inp = make_inputs(wl, "cuda")
    prob = Problem.from_inputs(wl, inp)
    out = torch.full((wl.rows, wl.N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    prob.run_gpu(out=out)
    torch.cuda.synchronize()
    rows = prob.sample_rows(per_group_random=1, seed=wl.seed, cap=64)
    got = bits_of(out[torch.from_numpy(rows).cuda()]).reshape(rows.size, wl.N)
    ref, ab = prob.oracle_rows(orc, rows)
    compare(got.ravel(), ref.ravel(), ab.ravel(), name)
    _no_tile_skipped(out, prob.owned_rows_mask(), name)
    assert fx.device_status() == 0
    del inp, prob, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["n3_ragged_n_m1024", "n4_ragged_k_wgrad"])
def test_full_size_ragged_sampled(orc, name):
    # ragged layouts at full size through the C ABI, in the benchmark's plan; sampled output
    # rows compared in full (every column / every group's slab row)
    from parity_util import abs_codes
    wl = workloads()[name]
    inp = make_inputs(wl, "cuda")
    G, M = wl.G, wl.rows
    st = torch.cuda.current_stream().cuda_stream
    if wl.layout == "ragged_n":
        out = torch.full((M, wl.N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        s = fx.mslkb_f8f8bf16_rowwise_grouped_n_offsets(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), G, M, wl.N,
            wl.K, st)
        rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(wl.seed)
                                         .integers(0, M, 14)])).astype(np.int64)
    else:
        out = torch.full((G * M, wl.N), 0x7E7E, dtype=torch.int16,
                         device="cuda").view(torch.bfloat16)
        s = fx.mslkb_f8f8bf16_rowwise_grouped_k_offsets(
            inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
            inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), G, M, wl.N,
            wl.K, st)
        rng = np.random.default_rng(wl.seed)
        rows = np.unique(np.concatenate([[g * M, g * M + M - 1, g * M + rng.integers(0, M)]
                                         for g in range(G)])).astype(np.int64)
    assert s == fx.MSLKB_OK, fx.mslkb_status_string(s)
    torch.cuda.synchronize()
    got = bits_of(out[torch.from_numpy(rows).cuda()]).reshape(rows.size, wl.N)
    h = {k: v.cpu().numpy() for k, v in inp.items()}
    if wl.layout == "ragged_n":
        A = h["A"].reshape(G, M, wl.K)
        ref, _ = orc.n_offsets(A, h["B"], h["scale_a"].reshape(G, M), h["scale_b"], h["meta"],
                               rows=rows)
        ab, _ = orc.n_offsets(abs_codes(A), abs_codes(h["B"]), np.abs(h["scale_a"]).reshape(G, M),
                              np.abs(h["scale_b"]), h["meta"], rows=rows)
    else:
        ref, _ = orc.k_offsets(h["A"], h["B"], h["scale_a"].reshape(G, M),
                               h["scale_b"].reshape(G, wl.N), h["meta"], rows=rows)
        ab, _ = orc.k_offsets(abs_codes(h["A"]), abs_codes(h["B"]),
                              np.abs(h["scale_a"]).reshape(G, M),
                              np.abs(h["scale_b"]).reshape(G, wl.N), h["meta"], rows=rows)
    compare(got.ravel(), ref.ravel(), ab.ravel(), name)
    assert fx.device_status() == 0
    del inp, out
    torch.cuda.empty_cache()


def test_full_size_groupwise_sampled(orc):
    # the block-scaled workload at full size in the benchmark's plan; sampled rows in full
    from parity_util import abs_codes
    wl = workloads()["n5_groupwise_llama70b_m8192"]
    inp = make_inputs(wl, "cuda")
    out = torch.full((wl.rows, wl.N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    s = fx.mslkb_f8f8bf16_groupwise_grouped_stacked(
        inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
        inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.rows, wl.G, wl.N,
        wl.K, torch.cuda.current_stream().cuda_stream)
    assert s == fx.MSLKB_OK, fx.mslkb_status_string(s)
    torch.cuda.synchronize()
    off = np.concatenate([[0], np.cumsum(wl.meta)])
    rng = np.random.default_rng(wl.seed)
    rows = np.unique(np.concatenate([[off[g], off[g + 1] - 1, rng.integers(off[g], off[g + 1])]
                                     for g in range(wl.G) if off[g + 1] > off[g]])).astype(np.int64)
    got = bits_of(out[torch.from_numpy(rows).cuda()]).reshape(rows.size, wl.N)
    h = {k: v.cpu().numpy() for k, v in inp.items()}
    ref, _ = orc.blockwise_stacked(h["A"], h["B"], h["scale_a"], h["scale_b"], h["meta"],
                                   rows=rows)
    ab, _ = orc.blockwise_stacked(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["scale_a"]),
                                  np.abs(h["scale_b"]), h["meta"], rows=rows)
    compare(got.ravel(), ref.ravel(), ab.ravel(), wl.name)
    _no_tile_skipped(out, np.ones(wl.rows, bool), wl.name)
    assert fx.device_status() == 0
    del inp, out
    torch.cuda.empty_cache()


def test_full_size_groupwise_decode_sampled(orc):
    # the block-scaled decode workload (swap-AB tiles split along K) at full size, all rows
    from parity_util import abs_codes
    wl = workloads()["n6_groupwise_llama70b_m16"]
    inp = make_inputs(wl, "cuda")
    out = torch.full((wl.rows, wl.N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    s = fx.mslkb_f8f8bf16_groupwise_grouped_stacked(
        inp["A"].data_ptr(), inp["B"].data_ptr(), inp["scale_a"].data_ptr(),
        inp["scale_b"].data_ptr(), inp["meta"].data_ptr(), out.data_ptr(), wl.rows, wl.G, wl.N,
        wl.K, torch.cuda.current_stream().cuda_stream)
    assert s == fx.MSLKB_OK, fx.mslkb_status_string(s)
    torch.cuda.synchronize()
    got = bits_of(out).reshape(wl.rows, wl.N)
    h = {k: v.cpu().numpy() for k, v in inp.items()}
    ref, _ = orc.blockwise_stacked(h["A"], h["B"], h["scale_a"], h["scale_b"], h["meta"])
    ab, _ = orc.blockwise_stacked(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["scale_a"]),
                                  np.abs(h["scale_b"]), h["meta"])
    compare(got.ravel(), ref.ravel(), ab.ravel(), wl.name)
    assert fx.device_status() == 0
    del inp, out
    torch.cuda.empty_cache()
