"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle on the same
bytes, and compare under the tolerance of the method's statement of parity:

    |gpu - ref| <= 2 * ulp_bf16(ref) + 1e-6 * |scale_a * scale_b| * sum_k |A[r,k] * B[g,n,k]|

where ref is the oracle's correctly rounded bf16 value and ulp_bf16(ref) is
2^(max(floor(log2|ref|), -126) - 7) (2^-133 at ref = 0).  The absolute term is computed
by the oracle itself on |codes| and |scales| (its bf16 result is within 2^-8 of the exact
sum; the bound is widened by 2^-7 to cover that).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bits_of(out: torch.Tensor) -> np.ndarray:
    return to_np(out.contiguous().view(torch.int16)).astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_float(bits)


def abs_codes(codes: np.ndarray) -> np.ndarray:
    """|x| of E4M3 codes: clear the sign bit (NaN codes stay NaN)."""
    return (codes & 0x7F).astype(np.uint8)


def compare(gpu_bits: np.ndarray, ref_bits: np.ndarray, abs_bits: np.ndarray, what=""):
    """Assert the tolerance element by element; returns a stats dict."""
    g = bf16_values(gpu_bits)
    r = bf16_values(ref_bits)
    a = bf16_values(abs_bits) * (1.0 + 2.0 ** -7)
    nan_r, nan_g = np.isnan(r), np.isnan(g)
    assert np.array_equal(nan_r, nan_g), f"{what}: NaN positions differ ({nan_r.sum()} vs {nan_g.sum()})"
    fin = ~nan_r
    inf_r = np.isinf(r) & fin
    assert np.array_equal(g[inf_r], r[inf_r]), f"{what}: infinities differ"
    m = fin & ~inf_r
    rr, gg, aa = r[m], g[m], a[m]
    ar = np.abs(rr)
    e = np.floor(np.log2(np.where(ar > 0, ar, 1.0)))
    e = np.maximum(e, -126.0)
    ulp = np.where(ar > 0, np.exp2(e - 7.0), 2.0 ** -133)
    tol = 2.0 * ulp + 1e-6 * aa
    err = np.abs(gg - rr)
    bad = err > tol
    stats = {
        "elements": int(m.sum()),
        "bit_exact": float(np.mean(gpu_bits[m] == ref_bits[m])) if m.any() else 1.0,
        "max_err_over_tol": float(np.max(err / tol)) if m.any() else 0.0,
        "max_ulp": float(np.max(err / ulp)) if m.any() else 0.0,
    }
    if bad.any():
        idx = np.nonzero(bad)[0][:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {int(m.sum())} elements outside tolerance; "
            f"first: gpu={gg[idx]}, ref={rr[idx]}, tol={tol[idx]}; stats={stats}")
    return stats


class Problem:
    """One problem held both on the GPU (torch) and on the host (numpy)."""

    def __init__(self, layout, A, B, sa, sb, meta, expected_m=0, total_M=None):
        self.layout = layout
        self.A, self.B, self.sa, self.sb, self.meta = A, B, sa, sb, meta
        self.expected_m = expected_m
        self.G, self.N, self.K = B.shape
        self.rows = A.shape[0] if total_M is None else total_M
        self._host = None

    @classmethod
    def from_numpy(cls, layout, A, B, sa, sb, meta, expected_m=0, device="cuda"):
        def T(x, dt):
            return torch.from_numpy(np.ascontiguousarray(x)).to(device=device, dtype=dt)
        if layout == "offsets":
            m = T(np.asarray(meta, np.int32), torch.int32)
        else:
            m = T(np.asarray(meta, np.int64), torch.int64)
        return cls(layout, T(A, torch.uint8), T(B, torch.uint8), T(sa, torch.float32),
                   T(sb, torch.float32), m, expected_m)

    @classmethod
    def from_inputs(cls, wl, inp):
        return cls(wl.layout, inp["A"], inp["B"], inp["scale_a"], inp["scale_b"], inp["meta"],
                   wl.expected_m)

    def host(self):
        if self._host is None:
            self._host = dict(A=to_np(self.A), B=to_np(self.B), sa=to_np(self.sa),
                              sb=to_np(self.sb).reshape(self.G, self.N), meta=to_np(self.meta))
        return self._host

    # -- the CUDA path ------------------------------------------------------------------
    def run_gpu(self, out=None, variant=None):
        if variant is not None:
            fx.mslkb_force_variant(fx.variant_index(variant) if isinstance(variant, str)
                                   else variant)
        try:
            if self.layout == "stacked":
                return fx.f8f8bf16_rowwise_grouped_stacked(self.A, self.B, self.sa, self.sb,
                                                           self.meta, out=out)
            if self.layout == "offsets":
                return fx.f8f8bf16_rowwise_grouped_offsets(self.A, self.B, self.sa, self.sb,
                                                           self.meta, out=out)
            if self.layout == "batched":
                E = self.expected_m
                res = fx.f8f8bf16_rowwise_grouped_batched(
                    self.A.view(self.G, E, self.K), self.B, self.sa, self.sb,
                    out=None if out is None else out.view(self.G, E, self.N))
                return res.view(self.G * E, self.N)
            return fx.f8f8bf16_rowwise_grouped_dynamic(self.A, self.B, self.sa, self.sb,
                                                       self.meta, out=out)
        finally:
            if variant is not None:
                fx.mslkb_force_variant(-1)

    # -- the oracle ---------------------------------------------------------------------
    def oracle_full(self, orc, poison=None):
        h = self.host()
        if self.layout == "offsets":
            ref, _ = orc.offsets(h["A"], h["B"], h["sa"], h["sb"], h["meta"], total_M=self.rows,
                                 out=poison)
            ab, _ = orc.offsets(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["sa"]),
                                np.abs(h["sb"]), h["meta"], total_M=self.rows)
        elif self.layout == "batched":
            ref = orc.batched(h["A"], h["B"], h["sa"], h["sb"])
            ab = orc.batched(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["sa"]),
                             np.abs(h["sb"]))
        elif self.layout == "stacked":
            ref, _ = orc.stacked(h["A"], h["B"], h["sa"], h["sb"], h["meta"], total_M=self.rows,
                                 out=poison)
            ab, _ = orc.stacked(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["sa"]),
                                np.abs(h["sb"]), h["meta"], total_M=self.rows)
        else:
            ref = orc.dynamic(h["A"], h["B"], h["sa"], h["sb"], h["meta"], self.expected_m)
            ab = orc.dynamic(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["sa"]),
                             np.abs(h["sb"]), h["meta"], self.expected_m)
        return ref, ab

    def oracle_rows(self, orc, rows):
        h = self.host()
        if self.layout in ("stacked", "offsets"):
            # sampled rows via the stacked oracle on the groups' row counts (the offsets
            # pin checks the two layouts agree bit for bit)
            cnt = np.array(self.counts(), np.int64)
            ref = orc.stacked_rows(h["A"], h["B"], h["sa"], h["sb"], cnt, rows)
            ab = orc.stacked_rows(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["sa"]),
                                  np.abs(h["sb"]), cnt, rows)
        else:
            zsi = h["meta"] if self.layout == "dynamic" else \
                np.full(self.G, self.expected_m, np.int64)
            ref = orc.dynamic_rows(h["A"], h["B"], h["sa"], h["sb"], zsi, self.expected_m, rows)
            ab = orc.dynamic_rows(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["sa"]),
                                  np.abs(h["sb"]), zsi, self.expected_m, rows)
        return ref, ab

    def counts(self):
        """Rows of each group before clamping (stacked-like layouts)."""
        h = self.host()
        if self.layout == "offsets":
            o = [int(x) for x in h["meta"]]
            return [o[g] - (o[g - 1] if g else 0) for g in range(len(o))]
        return [int(x) for x in h["meta"]]

    def owned_rows_mask(self):
        mask = np.zeros(self.rows, dtype=bool)
        if self.layout in ("stacked", "offsets"):
            off = 0
            for m in self.counts():
                m = max(0, min(m, self.rows - off))
                mask[off:off + m] = True
                off += m
        else:
            mask[:] = True
        return mask

    def sample_rows(self, per_group_random=2, seed=0, cap=None):
        """First and last row of every non-empty group (or slab) plus a few random rows."""
        rng = np.random.default_rng(seed)
        h = self.host()
        rows = []
        if self.layout in ("stacked", "offsets"):
            off = 0
            for m in self.counts():
                m = max(0, min(int(m), self.rows - off))
                if m > 0:
                    rows += [off, off + m - 1]
                    rows += list(off + rng.integers(0, m, size=per_group_random))
                off += m
        else:
            E = self.expected_m
            zsi = h["meta"] if self.layout == "dynamic" else [E] * self.G
            for g, v in enumerate(zsi):
                v = max(0, min(int(v), E))
                rows += [g * E, g * E + E - 1]
                if v > 0:
                    rows += [g * E + v - 1] + list(g * E + rng.integers(0, v, size=per_group_random))
                if v < E:
                    rows += [g * E + v]
        rows = np.unique(np.array(rows, dtype=np.int64))
        if cap is not None and rows.size > cap:
            rows = np.sort(rng.choice(rows, size=cap, replace=False))
        return rows
