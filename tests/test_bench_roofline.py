"""bench.py's roofline accounting on CPU: clock samples are parsed and assigned to timed
windows, the FP8 peak is chosen from the window's clock (burst above the clock of the
sustained measurement, sustained at or below it), and the fractions follow from the time
and the chosen peak."""
import datetime

import pytest

import bench
from fp8_rowwise_scaled_gb300.synthetic import workloads

PK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
      "clocks_under_load": {"sm_mhz_median": 1460.0}}


def _line(t, sm, power, cap=False):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    act = "Active" if cap else "Not Active"
    return f"{stamp}, 0, {sm}, 2070, {power}, 0x0, Not Active, Not Active, Not Active, {act}"


def test_samples_parse_and_fall_into_windows():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.025 * i, 1400 + 10 * i, 1000.0 + i, cap=(i == 3)) for i in range(10)]
    rows = bench.parse_smi_rows(lines + ["garbage", ""])
    assert len(rows) == 10
    assert rows[3]["reasons"] == {"sw_power_cap"}
    s = bench.summarize_clocks([r for r in rows if t0 + 0.05 <= r["t"] <= t0 + 0.1])
    assert s["samples"] == 3 and s["sm_mhz"] == 1430.0 and s["reasons"] == ["sw_power_cap"]


def test_idle_samples_do_not_count_as_load():
    t0 = 1_800_000_000.0
    rows = bench.parse_smi_rows([_line(t0, 345, 100.0), _line(t0 + 0.1, 2010, 900.0),
                                 _line(t0 + 0.2, 1990, 1200.0)])
    assert bench.summarize_clocks(rows)["sm_mhz"] == 2000.0


def test_peak_follows_the_clock():
    burst, sust, f = bench.fp8_peaks(PK)
    assert (burst, sust, f) == (3800.0, 3400.0, 1460.0)
    assert bench.fp8_peak_for_clock(PK, 2010.0)[0] == burst
    assert bench.fp8_peak_for_clock(PK, 1461.0)[0] == burst
    assert bench.fp8_peak_for_clock(PK, 1460.0)[0] == sust
    assert bench.fp8_peak_for_clock(PK, 1300.0)[0] == sust
    assert bench.fp8_peak_for_clock(PK, None)[0] == burst
    assert bench.fp8_peak_for_clock({"hbm_gbs": 1.0, "bf16_tflops": 2.0}, 1000.0)[0] == 4.0


@pytest.mark.parametrize("sm,peak", [(2010.0, 3800.0), (1400.0, 3400.0)])
def test_fraction_recomputes_from_time_and_peak(sm, peak):
    wl = workloads()["c4_llama405b"]
    t = 2.7e-3
    r = bench.roofline(wl, PK, t, sm)
    assert r["bound"] == "tensor" and r["p_fp8"] == peak
    assert r["frac"] == pytest.approx(wl.flops() / t / 1e12 / peak)
    assert r["frac_nominal"] == pytest.approx(wl.flops() / t / 1e12 / bench.FP8_NOMINAL_TFLOPS)
    assert r["frac_at_clock"] == pytest.approx(wl.flops() / t / 1e12 / (3400.0 * sm / 1460.0))


def test_hbm_bound_shape():
    wl = workloads()["c3_llama70b_m16"]
    t = 120e-6
    r = bench.roofline(wl, PK, t, 1500.0)
    assert r["bound"] == "hbm"
    assert r["frac"] == pytest.approx(wl.bytes() / t / 1e9 / PK["hbm_gbs"])
    assert r["frac_nominal"] == pytest.approx(wl.bytes() / t / 1e9 / bench.HBM_NOMINAL_GBS)


def test_compact_rows_name_every_column():
    class Clk:
        def window(self, t0, t1):
            return {"sm_mhz": 1500.0}
    wl = workloads()["c3_llama70b_m16"]
    row = bench.shape_row({"wl": wl, "us": 120.0, "window": (0, 1), "variant": "v"}, PK, Clk())
    assert len(row) == len(bench.PER_SHAPE_COLS)
    assert row[0] == wl.name and row[3] == "hbm" and row[6] == 1500
    err = bench.shape_row({"workload": "x", "error": "boom"}, PK, Clk())
    assert len(err) == len(bench.PER_SHAPE_COLS) and err[0] == "x"


def test_per_shape_rows_fit_the_tail_of_the_line():
    # the rows come last on the output line; with the planner's variants and numbers as wide
    # as the sweep's, they and their column names fit in its last 1500 characters
    import json
    import fp8_rowwise_scaled_gb300 as fx
    from fp8_rowwise_scaled_gb300 import build as fxbuild
    fxbuild.build()
    wls = workloads()
    rows = []
    for n in list(bench.SWEEP) + [bench.HEADLINE]:
        plan = bench.plan_for(fx, wls[n], 152)          # the planner's variant on 152 SMs
        rows.append(bench.compact_row(n, 3074.14, 2861.32, "tensor", 0.8335, 0.6358, 2070.0,
                                      fx.variant_name(plan.variant)))
    tail = json.dumps({"per_shape_cols": bench.PER_SHAPE_COLS, "per_shape": rows},
                      separators=(",", ":"))
    assert len(tail) < 1500, len(tail)
