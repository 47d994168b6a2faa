"""CPU oracle for the FP8 rowwise-scaled grouped GEMM (stacked, dynamic, offsets, batched,
ragged-N and ragged-K layouts) and its block-scaled (groupwise) stacked, dynamic and
batched variants.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline
leg are the only callers.  Nothing here imports the CUDA library or its package, and
the CUDA library does not import this.

Two independent implementations live here:

* ``oracle.c`` (loaded through ctypes, built with gcc on first use): the fp64 oracle.
  It decodes E4M3 codes, sums exact products in fp64, applies both rowwise scales once
  and rounds the exact result to bf16 with round-to-nearest-even.  It follows the
  operation defined in MSLK #471 "Back the FP8 rowwise grouped GEMM ops with FlyDSL on
  ROCm" (commit introducing the rowwise scaling scheme; PR Summary table for the
  stacked / dynamic layouts).
* ``bruteforce.py``: the same definition in exact rational arithmetic (pure Python),
  for tiny inputs only.

Every function takes and returns numpy arrays; bf16 results are returned as uint16 bit
patterns so that comparisons are exact.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

# Mutants compiled from oracle.c with -DORACLE_MUTANT=<id>; each plants one mistake.
MUTANTS = {
    1: "last K term dropped",
    2: "B read as [G, K, N] (transposed operand)",
    3: "scale_b of group 0 used for every group",
    4: "rounded through binary32 before bf16 (double rounding)",
    5: "E4M3 exponent bias 8 instead of 7",
    6: "E4M3 sign bit ignored",
    7: "stacked group prefix off by one row",
    8: "dynamic padding rows not written",
    9: "bf16 ties rounded away from zero",
    10: "scale_b not applied",
    11: "ragged-N: the slab of group 0 used for every group",
    12: "ragged-K: every group's slice read from k = 0",
    13: "block scaling: the scales of K block 0 used for every block",
    14: "block-scaled dynamic: scale_a of the slab-local row",
}


def lib_path(mutant: int = 0) -> str:
    return os.path.join(_BUILD, f"liboracle_m{mutant}.so")


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile oracle.c (optionally a mutant) into a shared library; returns its path."""
    out = lib_path(mutant)
    with _LOCK:
        if (not force and os.path.exists(out)
                and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
            return out
        os.makedirs(_BUILD, exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-shared",
               "-fPIC", f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True, capture_output=True)
        os.replace(tmp, out)
        return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_bf16_round.argtypes = [ctypes.c_double, ctypes.c_double]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_stacked_offsets.argtypes = [p, i64, i64, p]
    lib.oracle_stacked_offsets.restype = ctypes.c_int
    lib.oracle_stacked.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, ctypes.c_int]
    lib.oracle_stacked.restype = ctypes.c_int
    lib.oracle_stacked_rows.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p,
                                        ctypes.c_int]
    lib.oracle_stacked_rows.restype = ctypes.c_int
    lib.oracle_dynamic.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, ctypes.c_int]
    lib.oracle_dynamic.restype = None
    lib.oracle_dynamic_rows.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p,
                                        ctypes.c_int]
    lib.oracle_dynamic_rows.restype = None
    lib.oracle_offsets.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, ctypes.c_int]
    lib.oracle_offsets.restype = ctypes.c_int
    lib.oracle_batched.argtypes = [p, p, p, p, i64, i64, i64, i64, p, ctypes.c_int]
    lib.oracle_batched.restype = None
    lib.oracle_n_offsets.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p, ctypes.c_int]
    lib.oracle_n_offsets.restype = ctypes.c_int
    lib.oracle_k_offsets.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p, ctypes.c_int]
    lib.oracle_k_offsets.restype = ctypes.c_int
    lib.oracle_blockwise_stacked.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p,
                                             ctypes.c_int]
    lib.oracle_blockwise_stacked.restype = ctypes.c_int
    lib.oracle_blockwise_dynamic.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p,
                                             ctypes.c_int]
    lib.oracle_blockwise_dynamic.restype = ctypes.c_int
    lib.oracle_dot_int.argtypes = [p, p, i64]
    lib.oracle_dot_int.restype = ctypes.c_int64
    lib.oracle_dot.argtypes = [p, p, i64]
    lib.oracle_dot.restype = ctypes.c_double
    lib.oracle_bf16_round_array.argtypes = [p, p, i64, p]
    lib.oracle_bf16_round_array.restype = None
    lib.oracle_mutant_id.argtypes = []
    lib.oracle_mutant_id.restype = ctypes.c_int
    return lib


def load(mutant: int = 0) -> "Oracle":
    if mutant not in _LIBS:
        _LIBS[mutant] = _declare(ctypes.CDLL(build(mutant)))
    return Oracle(_LIBS[mutant])


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data if a.size else 0


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


class Oracle:
    """Typed numpy front end over one build of oracle.c."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib
        self.mutant = lib.oracle_mutant_id()

    # -- scalar pieces ------------------------------------------------------------
    def e4m3_to_double(self, code: int) -> float:
        return self.lib.oracle_e4m3_to_double(code & 0xFF)

    def decode_table(self) -> np.ndarray:
        return np.array([self.e4m3_to_double(c) for c in range(256)], dtype=np.float64)

    def bf16_round(self, hi: float, lo: float = 0.0) -> int:
        return int(self.lib.oracle_bf16_round(hi, lo))

    def bf16_round_array(self, hi, lo=None) -> np.ndarray:
        h = _c(hi, np.float64).ravel()
        lo_arr = None if lo is None else _c(lo, np.float64).ravel()
        out = np.empty(h.size, dtype=np.uint16)
        self.lib.oracle_bf16_round_array(_ptr(h), 0 if lo_arr is None else _ptr(lo_arr),
                                         h.size, _ptr(out))
        return out

    def dot(self, arow, brow) -> float:
        a = _c(arow, np.uint8)
        b = _c(brow, np.uint8)
        return float(self.lib.oracle_dot(_ptr(a), _ptr(b), a.size))

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(bits & 0xFFFF)

    def stacked_offsets(self, m_sizes, total_M: int):
        m = _c(m_sizes, np.int64)
        off = np.zeros(m.size + 1, dtype=np.int64)
        clamped = self.lib.oracle_stacked_offsets(_ptr(m), m.size, int(total_M), _ptr(off))
        return off, bool(clamped)

    def dot_int(self, arow, brow) -> int:
        a = _c(arow, np.uint8)
        b = _c(brow, np.uint8)
        return int(self.lib.oracle_dot_int(_ptr(a), _ptr(b), a.size))

    # -- whole problems -----------------------------------------------------------
    def stacked(self, A, B, scale_a, scale_b, m_sizes, total_M=None, out=None,
                threads: int = 0):
        """A [total_M, K] u8, B [G, N, K] u8, scale_a [total_M] f32, scale_b [G, N] f32,
        m_sizes [G] i64.  Returns (out [total_M, N] u16, clamped).  Rows past the last
        group keep the contents of ``out`` (zeros if ``out`` is None)."""
        A = _c(A, np.uint8)
        B = _c(B, np.uint8)
        G, N, K = B.shape
        if total_M is None:
            total_M = A.shape[0]
        sa = _c(scale_a, np.float32)
        sb = _c(scale_b, np.float32).reshape(G, N)
        m = _c(m_sizes, np.int64)
        assert m.size == G and A.shape == (total_M, K) and sa.size == total_M
        if out is None:
            out = np.zeros((total_M, N), dtype=np.uint16)
        else:
            out = _c(out, np.uint16).copy()
        clamped = self.lib.oracle_stacked(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(m),
                                          G, N, K, int(total_M), _ptr(out), int(threads))
        return out, bool(clamped)

    def stacked_rows(self, A, B, scale_a, scale_b, m_sizes, rows, threads: int = 0):
        """Full output rows ``rows`` of the stacked problem; 0xFFFF marks a row that
        belongs to no group."""
        A = _c(A, np.uint8)
        B = _c(B, np.uint8)
        G, N, K = B.shape
        total_M = A.shape[0]
        sa = _c(scale_a, np.float32)
        sb = _c(scale_b, np.float32).reshape(G, N)
        m = _c(m_sizes, np.int64)
        r = _c(rows, np.int64)
        out = np.zeros((r.size, N), dtype=np.uint16)
        self.lib.oracle_stacked_rows(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(m), G, N,
                                     K, total_M, _ptr(r), r.size, _ptr(out), int(threads))
        return out

    def dynamic(self, A, B, scale_a, scale_b, zsi, expected_m: int, threads: int = 0):
        """A [G*E, K] u8, B [G, N, K] u8, scale_a [G*E] f32, scale_b [G, N] f32,
        zsi [G] i64.  Returns out [G*E, N] u16 with padding rows +0.0."""
        A = _c(A, np.uint8)
        B = _c(B, np.uint8)
        G, N, K = B.shape
        E = int(expected_m)
        sa = _c(scale_a, np.float32)
        sb = _c(scale_b, np.float32).reshape(G, N)
        z = _c(zsi, np.int64)
        assert z.size == G and A.shape == (G * E, K) and sa.size == G * E
        out = np.full((G * E, N), 0xABCD, dtype=np.uint16)
        self.lib.oracle_dynamic(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(z), G, E, N, K,
                                _ptr(out), int(threads))
        return out

    def offsets(self, A, B, scale_a, scale_b, offsets, total_M=None, out=None,
                threads: int = 0):
        """Offsets layout: offsets [G] int32 inclusive prefix (group g owns rows
        [offsets[g-1], offsets[g])).  Returns (out [total_M, N] u16, clamped)."""
        A = _c(A, np.uint8)
        B = _c(B, np.uint8)
        G, N, K = B.shape
        if total_M is None:
            total_M = A.shape[0]
        sa = _c(scale_a, np.float32)
        sb = _c(scale_b, np.float32).reshape(G, N)
        o = _c(offsets, np.int32)
        assert o.size == G and A.shape == (total_M, K) and sa.size == total_M
        out = np.zeros((total_M, N), dtype=np.uint16) if out is None else \
            _c(out, np.uint16).copy()
        clamped = self.lib.oracle_offsets(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(o), G, N,
                                          K, int(total_M), _ptr(out), int(threads))
        return out, bool(clamped)

    def batched(self, A, B, scale_a, scale_b, threads: int = 0):
        """Batched layout: A [G*M, K] (or [G, M, K]), every row of every slab computed.
        Returns out [G*M, N] u16."""
        B = _c(B, np.uint8)
        G, N, K = B.shape
        sa = _c(scale_a, np.float32)
        M = sa.size // G if G else 0
        A = _c(A, np.uint8).reshape(G * M, K)
        sb = _c(scale_b, np.float32).reshape(G, N)
        assert A.shape[0] == G * M and sa.size == G * M
        out = np.full((G * M, N), 0xABCD, dtype=np.uint16)
        self.lib.oracle_batched(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), G, M, N, K, _ptr(out),
                                int(threads))
        return out

    def dynamic_rows(self, A, B, scale_a, scale_b, zsi, expected_m: int, rows,
                     threads: int = 0):
        A = _c(A, np.uint8)
        B = _c(B, np.uint8)
        G, N, K = B.shape
        E = int(expected_m)
        sa = _c(scale_a, np.float32)
        sb = _c(scale_b, np.float32).reshape(G, N)
        z = _c(zsi, np.int64)
        r = _c(rows, np.int64)
        out = np.zeros((r.size, N), dtype=np.uint16)
        self.lib.oracle_dynamic_rows(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(z), G, E,
                                     N, K, _ptr(r), r.size, _ptr(out), int(threads))
        return out

    def n_offsets(self, A, B, scale_a, scale_b, offsets, rows=None, out=None,
                  threads: int = 0):
        """Ragged-N layout: A [G, M, K] u8, B [total_N, K] u8, scale_a [G, M] f32,
        scale_b [total_N] f32, offsets [G] int32 inclusive prefix over N.  Returns
        (out [M, total_N] u16 -- or the chosen ``rows`` of it --, clamped).  Columns past
        the last group keep the contents of ``out`` (zeros if None)."""
        B = _c(B, np.uint8)
        total_N, K = B.shape
        o = _c(offsets, np.int32)
        G = o.size
        sa = _c(scale_a, np.float32).ravel()
        M = sa.size // G if G else 0
        A = _c(A, np.uint8).reshape(G * M, K)
        sb = _c(scale_b, np.float32).ravel()
        assert sb.size == total_N and sa.size == G * M
        r = None if rows is None else _c(rows, np.int64)
        n_out = M if r is None else r.size
        if out is None:
            out = np.zeros((n_out, total_N), dtype=np.uint16)
        else:
            out = _c(out, np.uint16).reshape(n_out, total_N).copy()
        clamped = self.lib.oracle_n_offsets(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(o), G, M,
                                            total_N, K, 0 if r is None else _ptr(r),
                                            0 if r is None else r.size, _ptr(out), int(threads))
        return out, bool(clamped)

    def k_offsets(self, A, B, scale_a, scale_b, offsets, rows=None, threads: int = 0):
        """Ragged-K layout: A [M, total_K] u8, B [N, total_K] u8, scale_a [G, M] f32,
        scale_b [G, N] f32, offsets [G] int32 inclusive prefix over K.  Returns (out
        [G*M, N] u16 -- or the chosen slab ``rows`` of it --, clamped)."""
        A = _c(A, np.uint8)
        B = _c(B, np.uint8)
        M, total_K = A.shape
        N = B.shape[0]
        o = _c(offsets, np.int32)
        G = o.size
        sa = _c(scale_a, np.float32).ravel()
        sb = _c(scale_b, np.float32).ravel()
        assert B.shape == (N, total_K) and sa.size == G * M and sb.size == G * N
        r = None if rows is None else _c(rows, np.int64)
        n_out = G * M if r is None else r.size
        out = np.full((n_out, N), 0xABCD, dtype=np.uint16)
        clamped = self.lib.oracle_k_offsets(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(o), G, M,
                                            N, total_K, 0 if r is None else _ptr(r),
                                            0 if r is None else r.size, _ptr(out), int(threads))
        return out, bool(clamped)

    def blockwise_stacked(self, A, B, scale_a, scale_b, m_sizes, total_M=None, rows=None,
                          out=None, threads: int = 0):
        """Block-scaled stacked layout (blocks of 128 along K and N): A [total_M, K] u8,
        B [G, N, K] u8, scale_a [total_M, K/128] f32, scale_b [G, N/128, K/128] f32,
        m_sizes [G] i64.  Returns (out [total_M, N] u16 -- or the chosen ``rows`` of it,
        0xFFFF for a row of no group --, clamped)."""
        A = _c(A, np.uint8)
        B = _c(B, np.uint8)
        G, N, K = B.shape
        if total_M is None:
            total_M = A.shape[0]
        sa = _c(scale_a, np.float32).ravel()
        sb = _c(scale_b, np.float32).ravel()
        m = _c(m_sizes, np.int64)
        assert K % 128 == 0 and N % 128 == 0
        assert sa.size == total_M * (K // 128) and sb.size == G * (N // 128) * (K // 128)
        r = None if rows is None else _c(rows, np.int64)
        n_out = total_M if r is None else r.size
        if out is None:
            out = np.zeros((n_out, N), dtype=np.uint16)
        else:
            out = _c(out, np.uint16).reshape(n_out, N).copy()
        clamped = self.lib.oracle_blockwise_stacked(
            _ptr(A), _ptr(B), _ptr(sa), _ptr(sb), _ptr(m), G, N, K, int(total_M),
            0 if r is None else _ptr(r), 0 if r is None else r.size, _ptr(out), int(threads))
        assert clamped != -2
        return out, bool(clamped)


    def blockwise_dynamic(self, A, B, scale_a, scale_b, zsi, expected_m: int, rows=None,
                          threads: int = 0):
        """Block-scaled dynamic layout (blocks of 128 along K and N): A [G*E, K] u8,
        B [G, N, K] u8, scale_a [G*E, K/128] f32, scale_b [G, N/128, K/128] f32, zsi [G]
        i64 (None: every slab row valid -- the batched layout).  Returns out [G*E, N] u16,
        or the chosen slab ``rows`` of it; padding rows are +0.0."""
        A = _c(A, np.uint8)
        B = _c(B, np.uint8)
        G, N, K = B.shape
        E = int(expected_m)
        sa = _c(scale_a, np.float32).ravel()
        sb = _c(scale_b, np.float32).ravel()
        assert K % 128 == 0 and N % 128 == 0
        assert sa.size == G * E * (K // 128) and sb.size == G * (N // 128) * (K // 128)
        z = None if zsi is None else _c(zsi, np.int64)
        r = None if rows is None else _c(rows, np.int64)
        n_out = G * E if r is None else r.size
        out = np.zeros((n_out, N), dtype=np.uint16)
        rc = self.lib.oracle_blockwise_dynamic(
            _ptr(A), _ptr(B), _ptr(sa), _ptr(sb), 0 if z is None else _ptr(z), G, E, N, K,
            0 if r is None else _ptr(r), 0 if r is None else r.size, _ptr(out), int(threads))
        assert rc == 0
        return out

    def blockwise_batched(self, A, B, scale_a, scale_b, rows=None, threads: int = 0):
        """Block-scaled batched layout: every group owns a full slab of A.shape[0] / G rows."""
        G = B.shape[0]
        return self.blockwise_dynamic(A, B, scale_a, scale_b, None, A.shape[0] // G, rows,
                                      threads)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (bf16 is the upper half of binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
