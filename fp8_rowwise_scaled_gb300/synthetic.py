"""Seeded synthetic inputs for the FP8 rowwise-scaled grouped GEMM.

This module holds no part of the GEMM's arithmetic.  It only makes inputs, and it is
the one module that both the CUDA path's tests/benchmark and the CPU oracle's tests
draw inputs from.

Group metadata (m_sizes, zero_start_index_M) comes from splitmix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014), so it is the
same on every machine.  Each 64-bit output x gives the uniform u = (x >> 11) * 2^-53.

Bulk data is standard normal fp32 from torch.randn under a seeded torch.Generator on
the chosen device.  It is quantised per row to OCP FP8 E4M3 with scale = amax / 448:
one scale per row of A and one per (group, n) row of B, both kept in fp32.  A row whose
amax is 0 gets scale 1 and all-zero codes.  CPU and GPU generators give different
streams; every consumer reads back the bytes it was actually given.

The workloads are the five shape families the method was swept on (MSLK #471 "Back the
FP8 rowwise grouped GEMM ops with FlyDSL on ROCm": DS-V3, llama3-70b and llama3-405b
shape sweeps, plus the padded layout's test of empty, partial and full groups).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

MASK64 = (1 << 64) - 1
E4M3_MAX = 448.0


def splitmix64(state: int):
    """Generator of splitmix64 outputs from a 64-bit seed."""
    x = state & MASK64
    while True:
        x = (x + 0x9E3779B97F4A7C15) & MASK64
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def uniforms(seed: int, count: int) -> list[float]:
    g = splitmix64(seed)
    return [(next(g) >> 11) * 2.0 ** -53 for _ in range(count)]


def zipf_probs(G: int, s: float) -> list[float]:
    w = [(j + 1) ** (-s) for j in range(G)]
    tot = sum(w)
    return [x / tot for x in w]


def multinomial_counts(seed: int, total: int, probs: list[float]) -> list[int]:
    """``total`` independent categorical draws by inverse CDF over fp64 cumulative
    probabilities; returns the count per category."""
    cdf = []
    acc = 0.0
    for p in probs:
        acc += p
        cdf.append(acc)
    counts = [0] * len(probs)
    for u in uniforms(seed, total):
        j = 0
        while j < len(cdf) - 1 and u >= cdf[j]:
            j += 1
        counts[j] += 1
    return counts


@dataclass(frozen=True)
class Workload:
    """One problem: layout, sizes and group metadata (m_sizes or zero_start_index_M)."""
    name: str
    layout: str            # "stacked", "dynamic", "offsets", "batched", "ragged_n", "ragged_k",
                           # "groupwise" (stacked, block scales), "groupwise_dynamic",
                           # "groupwise_batched" (slabs, block scales)
    G: int
    N: int                 # output columns (total_N for ragged_n)
    K: int                 # contraction length (total_K for ragged_k)
    rows: int              # total_M (stacked), G * expected_m (dynamic), M (ragged)
    meta: tuple            # m_sizes (stacked), zero_start_index_M (dynamic), int32
                           # inclusive offsets (offsets; over N for ragged_n, over K for
                           # ragged_k); empty (batched)
    seed: int
    expected_m: int = 0    # dynamic only
    note: str = ""
    tags: tuple = field(default_factory=tuple)

    @property
    def total_M(self) -> int:
        return self.rows

    def ranges(self) -> list:
        """Ragged layouts: each group's [start, end) columns (ragged_n) or K slice
        (ragged_k), from the inclusive offsets."""
        out, start = [], 0
        total = self.N if self.layout == "ragged_n" else self.K
        for g in range(self.G):
            c = max(0, min(self.meta[g] - (self.meta[g - 1] if g else 0), total - start))
            out.append((start, start + c))
            start += c
        return out

    def counts(self) -> list:
        """Rows of each group (ragged layouts: the M rows of every group)."""
        if self.layout in ("ragged_n", "ragged_k"):
            return [self.rows] * self.G
        if self.layout in ("stacked", "groupwise"):
            return [max(0, m) for m in self.meta]
        if self.layout == "offsets":
            return [max(0, self.meta[g] - (self.meta[g - 1] if g else 0))
                    for g in range(self.G)]
        if self.layout in ("batched", "groupwise_batched"):
            return [self.expected_m] * self.G
        return [max(0, min(v, self.expected_m)) for v in self.meta]

    @property
    def slabs(self) -> bool:
        """True for the layouts whose groups own fixed slabs of expected_m rows."""
        return self.layout in ("dynamic", "batched", "groupwise_dynamic", "groupwise_batched")

    @property
    def block_scaled(self) -> bool:
        """True for the block-scaled (groupwise) layouts."""
        return self.layout.startswith("groupwise")

    def valid_rows(self) -> int:
        return sum(self.counts())

    def nonempty_groups(self) -> int:
        return sum(1 for c in self.counts() if c > 0)

    def flops(self) -> int:
        """Algorithmic flops: 2 * (valid rows) * N * K; ragged layouts: 2 * M * (owned
        columns) * K, or 2 * M * N * (sum of the K slices)."""
        if self.layout in ("ragged_n", "ragged_k"):
            owned = sum(e - s for s, e in self.ranges())
            return 2 * self.rows * owned * (self.K if self.layout == "ragged_n" else self.N)
        return 2 * self.valid_rows() * self.N * self.K

    def bytes(self) -> int:
        """Algorithmic HBM bytes of one call: every valid row of A and its scale, the
        weights and scales of non-empty groups only, the metadata, and the output
        (owned rows for stacked; the whole slab for dynamic, whose padding is
        written with zeros)."""
        if self.layout == "ragged_n":   # A slabs, B rows and scales, owned output columns
            owned = sum(e - s for s, e in self.ranges())
            return (self.G * self.rows * (self.K + 4) + self.N * (self.K + 4) + 4 * self.G
                    + 2 * self.rows * owned)
        if self.layout == "ragged_k":   # A and B once, scales, a whole slab per group
            return (self.rows * self.K + self.N * self.K + 4 * self.G * (self.rows + self.N)
                    + 4 * self.G + 2 * self.G * self.rows * self.N)
        v = self.valid_rows()
        nz = self.nonempty_groups()
        if self.block_scaled:   # scales per (row, K block) and per 128 x 128 block
            nkb = self.K // 128
            b = (v * (self.K + 4 * nkb) + nz * (self.N * self.K + 4 * (self.N // 128) * nkb)
                 + (8 * self.G if self.layout != "groupwise_batched" else 0))
            return b + 2 * (self.G * self.expected_m if self.slabs else v) * self.N
        b = v * self.K + 4 * v + nz * self.N * self.K + 4 * nz * self.N + 8 * self.G
        if self.slabs:
            b += 2 * self.G * self.expected_m * self.N
        else:
            b += 2 * v * self.N
        return b


def _stacked(name, cfg, sub, G, N, K, m_sizes, note="", tags=()):
    return Workload(name=name, layout="stacked", G=G, N=N, K=K, rows=sum(m_sizes),
                    meta=tuple(int(m) for m in m_sizes), seed=1000 * cfg + sub, note=note,
                    tags=tuple(tags))


def _inclusive(counts) -> list:
    out, acc = [], 0
    for c in counts:
        acc += int(c)
        out.append(acc)
    return out


def workloads() -> dict[str, Workload]:
    """The five configurations, by name.  Seeds are 1000 * config + sub-case."""
    w: dict[str, Workload] = {}
    # 0: small stacked case with an empty group
    w["c0_stacked_small"] = _stacked("c0_stacked_small", 0, 0, 4, 256, 512, [0, 3, 17, 44],
                                     "G=4, m_sizes=[0,3,17,44], N=256, K=512", ("parity",))
    # 1: dynamic (padded) layout with an empty and a full group, K and N tails
    G, E = 8, 128
    u = uniforms(1000 * 1 + 0, G)
    zsi = [1 + int(127 * x) for x in u]
    zsi[0] = 0
    zsi[7] = 128
    w["c1_dynamic_tails"] = Workload(
        name="c1_dynamic_tails", layout="dynamic", G=G, N=1000, K=1000, rows=G * E,
        meta=tuple(zsi), seed=1000, expected_m=E,
        note="G=8, expected_m=128, N=K=1000, zero_start_index_M uniform [1,127], "
             "group 0 empty, group 7 full", tags=("parity",))
    # 2: DS-V3-shaped MoE, 32 local experts, Zipf(1.1) routing of 8192 token-rows
    m2 = multinomial_counts(1000 * 2 + 0, 8192, zipf_probs(32, 1.1))
    w["c2a_dsv3_gate_up"] = _stacked("c2a_dsv3_gate_up", 2, 1, 32, 4096, 7168, m2,
                                     "DS-V3 gate_up: G=32, total_M=8192 Zipf(1.1), "
                                     "N=4096, K=7168", ("perf",))
    w["c2b_dsv3_down"] = _stacked("c2b_dsv3_down", 2, 2, 32, 7168, 2048, m2,
                                  "DS-V3 down: G=32, total_M=8192 Zipf(1.1), N=7168, K=2048",
                                  ("perf",))
    # 3: llama3-70b-shaped sweep, uniform routing over 16 groups
    for i, tm in enumerate([1, 16, 128, 1024, 8192]):
        m3 = multinomial_counts(1000 * 3 + i, tm, [1.0 / 16] * 16)
        nm = f"c3_llama70b_m{tm}"
        w[nm] = _stacked(nm, 3, i, 16, 8192, 8192, m3,
                         f"llama3-70b: G=16, N=K=8192, total_M={tm} uniform", ("perf",))
    # NEXT rows: the same llama3-70b total_M = 8192 routing given as int32 inclusive
    # offsets, and a batched (every slab full) problem of the same size
    m3 = w["c3_llama70b_m8192"].meta
    incl, acc = [], 0
    for m in m3:
        acc += m
        incl.append(acc)
    w["n2_offsets_llama70b_m8192"] = Workload(
        name="n2_offsets_llama70b_m8192", layout="offsets", G=16, N=8192, K=8192, rows=acc,
        meta=tuple(incl), seed=1000 * 3 + 4,
        note="llama3-70b total_M=8192 routing as int32 inclusive offsets", tags=("perf",))
    w["n1_batched_llama70b_m512"] = Workload(
        name="n1_batched_llama70b_m512", layout="batched", G=16, N=8192, K=8192,
        rows=16 * 512, meta=(), seed=1000 * 5 + 0, expected_m=512,
        note="batched: G=16 full slabs of 512 rows, N=K=8192", tags=("perf",))
    # NEXT-3: ragged N (the weights of 16 groups as one [16384, 8192] matrix split by a
    # uniform multinomial over columns, 1024 rows per group's slab) and ragged K (a
    # weight-gradient shape: 32768 tokens sliced over 16 groups in steps of 16, M = N =
    # 4096 per group)
    cn = multinomial_counts(1000 * 6 + 0, 16384, [1.0 / 16] * 16)
    w["n3_ragged_n_m1024"] = Workload(
        name="n3_ragged_n_m1024", layout="ragged_n", G=16, N=16384, K=8192, rows=1024,
        meta=tuple(_inclusive(cn)), seed=1000 * 6 + 0,
        note="ragged N: G=16 slabs of M=1024 rows, total_N=16384 multinomial, K=8192",
        tags=("perf",))
    ck = [16 * c for c in multinomial_counts(1000 * 7 + 0, 32768 // 16, [1.0 / 16] * 16)]
    w["n4_ragged_k_wgrad"] = Workload(
        name="n4_ragged_k_wgrad", layout="ragged_k", G=16, N=4096, K=32768, rows=4096,
        meta=tuple(_inclusive(ck)), seed=1000 * 7 + 0,
        note="ragged K: G=16 slices of 32768 (steps of 16), M=N=4096", tags=("perf",))
    # NEXT-4: block scaling (128 x 128 weight blocks, 1 x 128 activation blocks) on the
    # llama3-70b total_M = 8192 routing
    w["n5_groupwise_llama70b_m8192"] = Workload(
        name="n5_groupwise_llama70b_m8192", layout="groupwise", G=16, N=8192, K=8192,
        rows=sum(m3), meta=tuple(m3), seed=1000 * 8 + 0,
        note="block-scaled: llama3-70b total_M=8192 routing, N=K=8192, 128-blocks",
        tags=("perf",))
    m16 = w["c3_llama70b_m16"].meta
    w["n6_groupwise_llama70b_m16"] = Workload(
        name="n6_groupwise_llama70b_m16", layout="groupwise", G=16, N=8192, K=8192,
        rows=sum(m16), meta=tuple(m16), seed=1000 * 8 + 1,
        note="block-scaled decode: llama3-70b total_M=16 routing, N=K=8192, 128-blocks",
        tags=("perf",))
    # NEXT-4 on the slab layouts: a batched problem of the n1 size, and a DS-V3 decode step
    # (256 routed token-rows, Zipf(1.1) over 32 experts, slabs of capacity 32 -- counts
    # above the capacity are clamped, as zero_start_index_M entries are)
    w["n7_groupwise_batched_llama70b_m512"] = Workload(
        name="n7_groupwise_batched_llama70b_m512", layout="groupwise_batched", G=16, N=8192,
        K=8192, rows=16 * 512, meta=(), seed=1000 * 8 + 2, expected_m=512,
        note="block-scaled batched: G=16 full slabs of 512 rows, N=K=8192, 128-blocks",
        tags=("perf",))
    z8 = multinomial_counts(1000 * 8 + 3, 256, zipf_probs(32, 1.1))
    w["n8_groupwise_dynamic_dsv3_m256"] = Workload(
        name="n8_groupwise_dynamic_dsv3_m256", layout="groupwise_dynamic", G=32, N=4096,
        K=7168, rows=32 * 32, meta=tuple(z8), seed=1000 * 8 + 3, expected_m=32,
        note="block-scaled dynamic: DS-V3 gate_up decode, 256 token-rows Zipf(1.1) over 32 "
             "slabs of 32 rows, N=4096, K=7168, 128-blocks", tags=("perf",))
    # 4: llama3-405b-shaped
    m4 = multinomial_counts(1000 * 4 + 0, 16384, [1.0 / 16] * 16)
    w["c4_llama405b"] = _stacked("c4_llama405b", 4, 0, 16, 16384, 16384, m4,
                                 "llama3-405b: G=16, N=K=total_M=16384 uniform", ("perf",))
    return w


# -------------------------------------------------------------------------------------
# bulk data
# -------------------------------------------------------------------------------------
def quantize_rows(x: torch.Tensor):
    """Per-row E4M3 quantisation of fp32 x [R, K]: returns (codes as uint8, scale fp32).

    scale = amax / 448 (fp32); codes = e4m3(clamp(x / scale, -448, 448)), using
    torch's round-to-nearest-even cast.  amax == 0 gives scale 1 and zero codes."""
    x = x.float()
    if x.shape[-1] == 0:
        return (torch.zeros(x.shape, dtype=torch.uint8, device=x.device),
                torch.ones(x.shape[:-1], dtype=torch.float32, device=x.device))
    amax = x.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (x / scale.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale.float()


def make_inputs(wl: Workload, device="cpu", chunk_rows: int = 8192):
    """Materialise a workload: A [rows, K] u8, B [G, N, K] u8, scale_a [rows] f32,
    scale_b [G, N] f32, meta [G] int64 (m_sizes or zero_start_index_M), all on
    ``device``.  Data comes from torch.randn under Generator(seed); A first, then B
    group by group, in chunks of ``chunk_rows`` rows to bound the fp32 temporaries."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    if wl.layout in ("ragged_n", "ragged_k"):
        return _make_ragged(wl, device, gen, chunk_rows)
    if wl.block_scaled:
        return _make_groupwise(wl, device, gen, chunk_rows)
    G, N, K, R = wl.G, wl.N, wl.K, wl.rows
    A = torch.empty((R, K), dtype=torch.uint8, device=device)
    sa = torch.empty((R,), dtype=torch.float32, device=device)
    for r0 in range(0, R, chunk_rows):
        r1 = min(R, r0 + chunk_rows)
        x = torch.randn((r1 - r0, K), generator=gen, device=device, dtype=torch.float32)
        A[r0:r1], sa[r0:r1] = quantize_rows(x)
    B = torch.empty((G, N, K), dtype=torch.uint8, device=device)
    sb = torch.empty((G, N), dtype=torch.float32, device=device)
    for g in range(G):
        for n0 in range(0, N, chunk_rows):
            n1 = min(N, n0 + chunk_rows)
            x = torch.randn((n1 - n0, K), generator=gen, device=device, dtype=torch.float32)
            B[g, n0:n1], sb[g, n0:n1] = quantize_rows(x)
    mdt = torch.int32 if wl.layout == "offsets" else torch.int64
    meta = torch.tensor(list(wl.meta), dtype=mdt, device=device)
    return {"A": A, "B": B, "scale_a": sa, "scale_b": sb, "meta": meta}


def _make_ragged(wl: Workload, device, gen, chunk_rows: int):
    """Ragged layouts.  ragged_n: A [G*M, K] with scale_a [G*M] per row, B [total_N, K]
    with scale_b [total_N] per row.  ragged_k: each group's K slice of A [M, total_K] and
    B [N, total_K] quantised on its own, one scale per (group, row): scale_a [G*M],
    scale_b [G*N].  meta: int32 inclusive offsets."""
    G, M = wl.G, wl.rows
    if wl.layout == "ragged_n":
        A = torch.empty((G * M, wl.K), dtype=torch.uint8, device=device)
        sa = torch.empty((G * M,), dtype=torch.float32, device=device)
        for r0 in range(0, G * M, chunk_rows):
            r1 = min(G * M, r0 + chunk_rows)
            x = torch.randn((r1 - r0, wl.K), generator=gen, device=device, dtype=torch.float32)
            A[r0:r1], sa[r0:r1] = quantize_rows(x)
        B = torch.empty((wl.N, wl.K), dtype=torch.uint8, device=device)
        sb = torch.empty((wl.N,), dtype=torch.float32, device=device)
        for n0 in range(0, wl.N, chunk_rows):
            n1 = min(wl.N, n0 + chunk_rows)
            x = torch.randn((n1 - n0, wl.K), generator=gen, device=device, dtype=torch.float32)
            B[n0:n1], sb[n0:n1] = quantize_rows(x)
    else:
        A = torch.zeros((M, wl.K), dtype=torch.uint8, device=device)
        B = torch.zeros((wl.N, wl.K), dtype=torch.uint8, device=device)
        sa = torch.ones((G * M,), dtype=torch.float32, device=device)
        sb = torch.ones((G * wl.N,), dtype=torch.float32, device=device)
        for g, (k0, k1) in enumerate(wl.ranges()):
            if k1 == k0:
                continue
            for (T, S, R) in ((A, sa, M), (B, sb, wl.N)):
                for r0 in range(0, R, chunk_rows):
                    r1 = min(R, r0 + chunk_rows)
                    x = torch.randn((r1 - r0, k1 - k0), generator=gen, device=device,
                                    dtype=torch.float32)
                    T[r0:r1, k0:k1], S[g * R + r0:g * R + r1] = quantize_rows(x)
    meta = torch.tensor(list(wl.meta), dtype=torch.int32, device=device)
    return {"A": A, "B": B, "scale_a": sa, "scale_b": sb, "meta": meta}


def _make_groupwise(wl: Workload, device, gen, chunk_rows: int):
    """Block-scaled layouts: A quantised per (row, 128-element K block) -> scale_a
    [rows, K/128] (rows = total_M, or G * expected_m for the slab layouts); B per 128 x 128
    block of each group -> scale_b [G, N/128, K/128]; meta: m_sizes or zero_start_index_M
    (int64; empty for the batched layout)."""
    G, N, K, R = wl.G, wl.N, wl.K, wl.rows
    nkb, nnb = K // 128, N // 128
    A = torch.empty((R, K), dtype=torch.uint8, device=device)
    sa = torch.empty((R, nkb), dtype=torch.float32, device=device)
    for r0 in range(0, R, chunk_rows):
        r1 = min(R, r0 + chunk_rows)
        x = torch.randn((r1 - r0, nkb, 128), generator=gen, device=device, dtype=torch.float32)
        q, s = quantize_rows(x)
        A[r0:r1], sa[r0:r1] = q.reshape(r1 - r0, K), s
    B = torch.empty((G, N, K), dtype=torch.uint8, device=device)
    sb = torch.empty((G, nnb, nkb), dtype=torch.float32, device=device)
    for g in range(G):
        for n0 in range(0, N, chunk_rows):
            n1 = min(N, n0 + chunk_rows)
            x = torch.randn((n1 - n0, K), generator=gen, device=device, dtype=torch.float32)
            blk = x.reshape((n1 - n0) // 128, 128, nkb, 128).permute(0, 2, 1, 3)
            blk = blk.reshape((n1 - n0) // 128, nkb, 128 * 128)
            q, s = quantize_rows(blk)   # one scale per 128 x 128 block
            B[g, n0:n1] = q.reshape((n1 - n0) // 128, nkb, 128, 128).permute(0, 2, 1, 3) \
                .reshape(n1 - n0, K)
            sb[g, n0 // 128:n1 // 128] = s
    meta = torch.tensor(list(wl.meta), dtype=torch.int64, device=device)
    return {"A": A, "B": B, "scale_a": sa, "scale_b": sb, "meta": meta}


def random_codes(shape, gen: torch.Generator, device="cpu", allow_nan: bool = False):
    """Uniformly random E4M3 byte codes (every code, NaN codes optional)."""
    c = torch.randint(0, 256, shape, generator=gen, device=device, dtype=torch.int32)
    if not allow_nan:
        nan = (c & 0x7F) == 0x7F
        c = torch.where(nan, c ^ 0x01, c)  # 0x7F -> 0x7E (448), 0xFF -> 0xFE (-448)
    return c.to(torch.uint8)
