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
    assert fx.device_status() == 0
    del inp, prob, out
    torch.cuda.empty_cache()
