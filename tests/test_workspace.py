"""Per-stream split-tile workspaces: the first call on a stream allocates one, and
mslkb_release_workspace frees it; the next call on that stream allocates a new one and
still matches the oracle (split swap-AB tiles, which use its partial sums and counters, and
CTA pairs, which take their tiles from its claim counter)."""
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


def _problem(G, N, K, m_sizes, seed):
    g = torch.Generator().manual_seed(seed)
    rows = int(sum(m_sizes))
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa = (torch.rand(rows, generator=g) + 0.5).numpy().astype(np.float32)
    sb = (torch.rand(G * N, generator=g) + 0.5).numpy().astype(np.float32).reshape(G, N)
    return Problem.from_numpy("stacked", A, B, sa, sb, m_sizes)


@pytest.mark.parametrize("case", ["split_swap", "cta_pairs"])
def test_release_then_call_again(case):
    if case == "split_swap":
        prob = _problem(8, 2048, 2048, [1, 0, 3, 2, 0, 1, 1, 2], 61)
        want = "stacked_swap_w128xa16_tma"
    else:
        prob = _problem(2, 8192, 256, [1100, 1000], 62)
        want = "stacked_pair256x256_tma"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = fx.mslkb_plan(0, prob.rows, prob.G, prob.N, prob.K, sms)
    assert fx.variant_name(plan.variant) == want
    orc = oracle.load(0)
    ref, ab = prob.oracle_full(orc)
    s = torch.cuda.Stream()
    base = fx.mslkb_workspace_count()
    for rnd in range(2):
        with torch.cuda.stream(s):
            out = prob.run_gpu()
        s.synchronize()
        assert fx.mslkb_workspace_count() == base + 1
        compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"{case}, round {rnd + 1}")
        fx.mslkb_release_workspace(s.cuda_stream)
        assert fx.mslkb_workspace_count() == base
    fx.mslkb_release_workspace(s.cuda_stream)  # nothing left to release: fine
    assert fx.device_status() == 0


def test_two_streams_at_once():
    """Two streams run split-tile problems at the same time, each on its own workspace
    (partial sums and arrival counters): interleaved launches on both streams, no
    synchronisation between them, and both results still match the oracle."""
    p1 = _problem(8, 2048, 2048, [1, 0, 3, 2, 0, 1, 1, 2], 63)
    p2 = _problem(4, 4096, 1024, [2, 1, 0, 3], 64)
    orc = oracle.load(0)
    refs = [p.oracle_full(orc) for p in (p1, p2)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [None, None]
    for _ in range(12):
        for i, (p, s) in enumerate(((p1, s1), (p2, s2))):
            with torch.cuda.stream(s):
                outs[i] = p.run_gpu()
    torch.cuda.synchronize()
    for i, (out, (ref, ab)) in enumerate(zip(outs, refs)):
        compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"stream {i + 1}")
    for s in (s1, s2):
        fx.mslkb_release_workspace(s.cuda_stream)
    assert fx.device_status() == 0


def test_host_threads_on_their_own_streams():
    # five host threads call the library at once (ctypes drops the GIL for the call), each on
    # a stream of its own: the first call on each stream creates its workspace under the
    # library's lock while the others plan and launch; every result must match the oracle
    import threading
    cases = [_problem(8, 2048, 2048, [1, 0, 3, 2, 0, 1, 1, 2], 71),      # split swap-AB
             _problem(8, 2048, 1024, [0, 2, 1, 1, 3, 0, 1, 4], 75),      # split swap-AB
             _problem(2, 8192, 256, [1100, 1000], 72),                   # CTA pairs, claims
             _problem(4, 520, 1000, [130, 0, 257, 64], 73),              # cp.async loader
             _problem(5, 392, 688, [130, 1, 257, 64, 17], 74)]           # 128-row tiles
    with_workspace = 3   # the split and pair plans; the others need none
    orc = oracle.load(0)
    refs = [p.oracle_full(orc) for p in cases]
    base = fx.mslkb_workspace_count()
    streams = [torch.cuda.Stream() for _ in cases]
    outs = [[None] * 6 for _ in cases]
    errors = []
    start = threading.Barrier(len(cases))

    def worker(i):
        try:
            torch.cuda.set_device(0)
            start.wait()
            with torch.cuda.stream(streams[i]):
                for r in range(6):
                    outs[i][r] = cases[i].run_gpu()
            streams[i].synchronize()
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a host thread did not finish"
    assert not errors, errors
    assert fx.mslkb_workspace_count() == base + with_workspace
    for i, (ref, ab) in enumerate(refs):
        for r in range(6):
            compare(bits_of(outs[i][r]).ravel(), ref.ravel(), ab.ravel(), f"thread {i} call {r}")
    for s in streams:
        fx.mslkb_release_workspace(s.cuda_stream)
    assert fx.mslkb_workspace_count() == base
    assert fx.device_status() == 0
