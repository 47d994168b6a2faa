"""fp8_rowwise_scaled_gb300 -- FP8 rowwise-scaled grouped GEMM for GB300 (sm_103a).

For each group g and every row r it owns:
    out[r, n] = bf16_rne(scale_a[r] * scale_b[g, n] * sum_k A[r, k] * B[g, n, k])
with A, B in float8_e4m3fn, fp32 scales and fp32 accumulation (MSLK #471 "Back the FP8
rowwise grouped GEMM ops with FlyDSL on ROCm": rowwise scaling scheme; stacked and
dynamic layouts in the PR Summary table).

All computation happens in libmslkb.so (hand-written sm_103a CUDA, C ABI in
include/mslkb.h).  This module only marshals arguments:

* ``mslkb_*`` functions mirror the C entry points one to one (raw integer pointers);
* ``f8f8bf16_rowwise_grouped_stacked`` / ``..._dynamic`` take torch CUDA tensors and
  call the same entry points on the current stream.

There is no fallback: if libmslkb.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmslkb.so")
CHECKED_LIB_PATH = os.path.join(_PKG, "libmslkb_checked.so")

MSLKB_OK, MSLKB_ERR_NULL, MSLKB_ERR_SHAPE, MSLKB_ERR_ALIGN, MSLKB_ERR_DEVICE, MSLKB_ERR_CUDA = range(6)
MSLKB_ERR_TOO_LARGE = 6
NOALLOC_SCRATCH_BYTES = 8 << 20
MSLKB_DEV_TIMEOUT = 0x1
MSLKB_DEV_MSIZES_CLAMPED = 0x2
MSLKB_DEV_BAD_SLICE = 0x4
MSLKB_DEV_BOUNDS = 0x8
MAX_GROUPS = 1024

_lib = None
_lock = threading.Lock()


class MslkbError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().mslkb_status_string(status).decode()
        if status == MSLKB_ERR_CUDA:
            msg += f" (cuda error {lib().mslkb_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [status {status}]")


class PlanInfo(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("swap_ab", ctypes.c_int32),
                ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("tma", ctypes.c_int32),
                ("copy_width", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("tiles_bound", ctypes.c_int64), ("split_k", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["variant_name"] = variant_name(self.variant)
        return d


def declare(L: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the argument and result types of the C entry points on a loaded copy of
    the library (libmslkb.so, or the checked build libmslkb_checked.so)."""
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    for name in ("mslkb_f8f8bf16_rowwise_grouped_stacked",
                 "mslkb_f8f8bf16_rowwise_grouped_dynamic",
                 "mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc",
                 "mslkb_f8f8bf16_groupwise_grouped_stacked"):
        fn = getattr(L, name)
        fn.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, p]
        fn.restype = ctypes.c_int
    L.mslkb_f8f8bf16_rowwise_grouped_offsets.argtypes = [p, p, p, p, p, p, i64, i64,
                                                         i64, i64, p]
    L.mslkb_f8f8bf16_rowwise_grouped_offsets.restype = ctypes.c_int
    L.mslkb_f8f8bf16_rowwise_grouped_batched.argtypes = [p, p, p, p, p, i64, i64, i64,
                                                         i64, p]
    L.mslkb_f8f8bf16_rowwise_grouped_batched.restype = ctypes.c_int
    L.mslkb_f8f8bf16_groupwise_grouped_dynamic.argtypes = [p, p, p, p, p, p, i64, i64,
                                                           i64, i64, p]
    L.mslkb_f8f8bf16_groupwise_grouped_dynamic.restype = ctypes.c_int
    L.mslkb_f8f8bf16_groupwise_grouped_batched.argtypes = [p, p, p, p, p, i64, i64, i64,
                                                           i64, p]
    L.mslkb_f8f8bf16_groupwise_grouped_batched.restype = ctypes.c_int
    for name in ("mslkb_f8f8bf16_rowwise_grouped_n_offsets",
                 "mslkb_f8f8bf16_rowwise_grouped_k_offsets"):
        fn = getattr(L, name)
        fn.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, p]
        fn.restype = ctypes.c_int
    L.mslkb_status_string.argtypes = [ctypes.c_int]
    L.mslkb_status_string.restype = ctypes.c_char_p
    L.mslkb_last_cuda_error.argtypes = []
    L.mslkb_last_cuda_error.restype = ctypes.c_int
    L.mslkb_get_device_status.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
    L.mslkb_get_device_status.restype = ctypes.c_int
    L.mslkb_plan.argtypes = [ctypes.c_int32, i64, i64, i64, i64, ctypes.c_int32, i64,
                             i64, ctypes.POINTER(PlanInfo)]
    L.mslkb_plan.restype = ctypes.c_int
    L.mslkb_num_variants.argtypes = []
    L.mslkb_num_variants.restype = ctypes.c_int32
    L.mslkb_variant_name.argtypes = [ctypes.c_int32]
    L.mslkb_variant_name.restype = ctypes.c_char_p
    L.mslkb_force_variant.argtypes = [ctypes.c_int32]
    L.mslkb_force_variant.restype = ctypes.c_int
    L.mslkb_variant_resources.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32)]
    L.mslkb_variant_resources.restype = ctypes.c_int
    L.mslkb_set_split_k.argtypes = [ctypes.c_int32]
    L.mslkb_set_split_k.restype = ctypes.c_int
    L.mslkb_set_accumulation_chunk.argtypes = [ctypes.c_int32]
    L.mslkb_set_accumulation_chunk.restype = ctypes.c_int
    L.mslkb_accumulation_chunk.argtypes = []
    L.mslkb_accumulation_chunk.restype = ctypes.c_int32
    L.mslkb_set_weight_prefetch.argtypes = [ctypes.c_int32]
    L.mslkb_set_weight_prefetch.restype = ctypes.c_int
    L.mslkb_test_speculate_from_next_launch.argtypes = [ctypes.c_void_p]
    L.mslkb_test_speculate_from_next_launch.restype = ctypes.c_int
    L.mslkb_set_wait_timeout_us.argtypes = [i64]
    L.mslkb_set_wait_timeout_us.restype = ctypes.c_int
    L.mslkb_test_stall_next_launch.argtypes = []
    L.mslkb_test_stall_next_launch.restype = ctypes.c_int
    L.mslkb_release_workspace.argtypes = [p]
    L.mslkb_release_workspace.restype = ctypes.c_int
    L.mslkb_workspace_count.argtypes = []
    L.mslkb_workspace_count.restype = ctypes.c_int32
    L.mslkb_version.argtypes = []
    L.mslkb_version.restype = ctypes.c_int32
    return L


def lib() -> ctypes.CDLL:
    """The loaded libmslkb.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m fp8_rowwise_scaled_gb300.build` (there is no fallback path)")
            _lib = declare(ctypes.CDLL(LIB_PATH))
    return _lib


# ---------------------------------------------------------------------------------------
# raw C entry points (integer pointers; stream = cudaStream_t as int, 0 = default stream)
# ---------------------------------------------------------------------------------------
def mslkb_f8f8bf16_rowwise_grouped_stacked(A, B, scale_a, scale_b, m_sizes, out, total_M, G,
                                           N, K, stream=0) -> int:
    return lib().mslkb_f8f8bf16_rowwise_grouped_stacked(A, B, scale_a, scale_b, m_sizes, out,
                                                        total_M, G, N, K, stream)


def mslkb_f8f8bf16_rowwise_grouped_dynamic(A, B, scale_a, scale_b, zero_start_index_M, out,
                                           G, expected_m, N, K, stream=0) -> int:
    return lib().mslkb_f8f8bf16_rowwise_grouped_dynamic(A, B, scale_a, scale_b,
                                                        zero_start_index_M, out, G, expected_m,
                                                        N, K, stream)


def mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc(A, B, scale_a, scale_b, m_sizes, out,
                                                   total_M, G, N, K, stream=0) -> int:
    """The stacked call with its split-tile scratch in a static device array: allocates
    nothing (for callers recording CUDA graphs or whose framework owns all memory)."""
    return lib().mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc(
        A, B, scale_a, scale_b, m_sizes, out, total_M, G, N, K, stream)


def mslkb_f8f8bf16_rowwise_grouped_offsets(A, B, scale_a, scale_b, offsets, out, total_M, G,
                                           N, K, stream=0) -> int:
    return lib().mslkb_f8f8bf16_rowwise_grouped_offsets(A, B, scale_a, scale_b, offsets, out,
                                                        total_M, G, N, K, stream)


def mslkb_f8f8bf16_rowwise_grouped_batched(A, B, scale_a, scale_b, out, G, M, N, K,
                                           stream=0) -> int:
    return lib().mslkb_f8f8bf16_rowwise_grouped_batched(A, B, scale_a, scale_b, out, G, M, N,
                                                        K, stream)


def mslkb_f8f8bf16_rowwise_grouped_n_offsets(A, B, scale_a, scale_b, offsets, out, G, M,
                                             total_N, K, stream=0) -> int:
    return lib().mslkb_f8f8bf16_rowwise_grouped_n_offsets(A, B, scale_a, scale_b, offsets, out,
                                                          G, M, total_N, K, stream)


def mslkb_f8f8bf16_rowwise_grouped_k_offsets(A, B, scale_a, scale_b, offsets, out, G, M, N,
                                             total_K, stream=0) -> int:
    return lib().mslkb_f8f8bf16_rowwise_grouped_k_offsets(A, B, scale_a, scale_b, offsets, out,
                                                          G, M, N, total_K, stream)


def mslkb_f8f8bf16_groupwise_grouped_stacked(A, B, scale_a, scale_b, m_sizes, out, total_M, G,
                                             N, K, stream=0) -> int:
    """Block-scaled stacked call: scale_a [total_M, K/128], scale_b [G, N/128, K/128]."""
    return lib().mslkb_f8f8bf16_groupwise_grouped_stacked(A, B, scale_a, scale_b, m_sizes, out,
                                                          total_M, G, N, K, stream)


def mslkb_f8f8bf16_groupwise_grouped_dynamic(A, B, scale_a, scale_b, zero_start_index_M, out,
                                             G, expected_m, N, K, stream=0) -> int:
    """Block-scaled dynamic call: scale_a [G*E, K/128], scale_b [G, N/128, K/128]."""
    return lib().mslkb_f8f8bf16_groupwise_grouped_dynamic(A, B, scale_a, scale_b,
                                                          zero_start_index_M, out, G,
                                                          expected_m, N, K, stream)


def mslkb_f8f8bf16_groupwise_grouped_batched(A, B, scale_a, scale_b, out, G, M, N, K,
                                             stream=0) -> int:
    """Block-scaled batched call: scale_a [G*M, K/128], scale_b [G, N/128, K/128]."""
    return lib().mslkb_f8f8bf16_groupwise_grouped_batched(A, B, scale_a, scale_b, out, G, M, N,
                                                          K, stream)


def mslkb_status_string(status: int) -> str:
    return lib().mslkb_status_string(status).decode()


def mslkb_get_device_status(stream=0) -> int:
    flags = ctypes.c_uint32(0)
    s = lib().mslkb_get_device_status(stream, ctypes.byref(flags))
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_get_device_status")
    return int(flags.value)


def mslkb_plan(layout: int, rows: int, G: int, N: int, K: int, num_sms: int,
               a_align: int = 256, b_align: int = 256) -> PlanInfo:
    info = PlanInfo()
    s = lib().mslkb_plan(layout, rows, G, N, K, num_sms, a_align, b_align, ctypes.byref(info))
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_plan")
    return info


def mslkb_num_variants() -> int:
    return lib().mslkb_num_variants()


def variant_name(i: int):
    n = lib().mslkb_variant_name(i)
    return n.decode() if n else None


def variant_index(name: str) -> int:
    for i in range(mslkb_num_variants()):
        if variant_name(i) == name:
            return i
    raise KeyError(name)


def mslkb_force_variant(i: int) -> None:
    s = lib().mslkb_force_variant(i)
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_force_variant")


def mslkb_variant_resources(i: int):
    """(CTAs per SM, registers per thread) of kernel variant i on the current device."""
    b, r = ctypes.c_int32(0), ctypes.c_int32(0)
    s = lib().mslkb_variant_resources(i, ctypes.byref(b), ctypes.byref(r))
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_variant_resources")
    return int(b.value), int(r.value)


def mslkb_set_split_k(enable: int) -> None:
    s = lib().mslkb_set_split_k(enable)
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_set_split_k")


def mslkb_set_accumulation_chunk(kblocks: int) -> None:
    s = lib().mslkb_set_accumulation_chunk(kblocks)
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_set_accumulation_chunk")


def mslkb_accumulation_chunk() -> int:
    return lib().mslkb_accumulation_chunk()


def mslkb_set_weight_prefetch(kblocks: int) -> None:
    s = lib().mslkb_set_weight_prefetch(kblocks)
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_set_weight_prefetch")


def mslkb_set_wait_timeout_us(us: int) -> None:
    s = lib().mslkb_set_wait_timeout_us(us)
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_set_wait_timeout_us")


def mslkb_test_speculate_from_next_launch(meta) -> None:
    """Test hook: the next launch's speculative weight prefetch reads `meta` (a device
    tensor laid out like that call's metadata) instead of the call's own metadata."""
    lib().mslkb_test_speculate_from_next_launch(ctypes.c_void_p(meta.data_ptr()))


def mslkb_release_workspace(stream=None) -> None:
    """Free the split-tile workspace of `stream` (default: the current torch stream) on
    the current device; the next call on that stream allocates a new one."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    s = lib().mslkb_release_workspace(ctypes.c_void_p(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "mslkb_release_workspace")


def mslkb_workspace_count() -> int:
    return lib().mslkb_workspace_count()


def mslkb_test_stall_next_launch() -> None:
    lib().mslkb_test_stall_next_launch()


def mslkb_version() -> int:
    return lib().mslkb_version()


# ---------------------------------------------------------------------------------------
# torch front end
# ---------------------------------------------------------------------------------------
def _check(t, name, dtypes, dim=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if dim is not None and t.dim() not in (dim if isinstance(dim, tuple) else (dim,)):
        raise ValueError(f"{name}: expected {dim} dims, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (strided views are not supported)")


def _fp8_types():
    import torch
    return (torch.float8_e4m3fn, torch.uint8)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def f8f8bf16_rowwise_grouped_stacked(XQ, WQ, x_scale, w_scale, m_sizes, out=None,
                                     stream=None):
    """XQ [total_M, K] e4m3, WQ [G, N, K] e4m3, x_scale [total_M] fp32, w_scale [G, N]
    fp32, m_sizes [G] int64 (all on one CUDA device) -> out [total_M, N] bf16.

    Rows past sum(m_sizes) are not written: a freshly allocated ``out`` is zeroed first
    so that no stale memory is returned there."""
    import torch
    _check(XQ, "XQ", _fp8_types(), 2)
    _check(WQ, "WQ", _fp8_types(), 3)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    _check(m_sizes, "m_sizes", (torch.int64,), 1)
    total_M, K = XQ.shape
    G, N, K2 = WQ.shape
    if K2 != K or x_scale.numel() != total_M or w_scale.numel() != G * N or m_sizes.numel() != G:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.zeros((total_M, N), dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,), 2)
        if tuple(out.shape) != (total_M, N):
            raise ValueError("out has the wrong shape")
    s = mslkb_f8f8bf16_rowwise_grouped_stacked(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(),
        m_sizes.data_ptr(), out.data_ptr(), total_M, G, N, K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_rowwise_grouped_stacked")
    return out


def f8f8bf16_rowwise_grouped_dynamic(XQ, WQ, x_scale, w_scale, zero_start_index_M, out=None,
                                     stream=None):
    """XQ [G, E, K] (or [G*E, K]) e4m3, WQ [G, N, K] e4m3, x_scale [G*E] fp32, w_scale
    [G, N] fp32, zero_start_index_M [G] int64 -> out [G, E, N] (or [G*E, N]) bf16, with
    every padding row of every slab +0.0."""
    import torch
    _check(XQ, "XQ", _fp8_types(), (2, 3))
    _check(WQ, "WQ", _fp8_types(), 3)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    _check(zero_start_index_M, "zero_start_index_M", (torch.int64,), 1)
    G, N, K = WQ.shape
    if XQ.dim() == 3:
        if XQ.shape[0] != G:
            raise ValueError("XQ and WQ disagree on G")
        E = XQ.shape[1]
        out_shape = (G, E, N)
    else:
        if G == 0 or XQ.shape[0] % G:
            raise ValueError("XQ rows must be G * expected_m")
        E = XQ.shape[0] // G
        out_shape = (G * E, N)
    if XQ.shape[-1] != K or x_scale.numel() != G * E or w_scale.numel() != G * N \
            or zero_start_index_M.numel() != G:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty(out_shape, dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,))
        if out.numel() != G * E * N:
            raise ValueError("out has the wrong size")
    s = mslkb_f8f8bf16_rowwise_grouped_dynamic(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(),
        zero_start_index_M.data_ptr(), out.data_ptr(), G, E, N, K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_rowwise_grouped_dynamic")
    return out


def f8f8bf16_rowwise_grouped_offsets(XQ, WQ, x_scale, w_scale, offsets, out=None,
                                     stream=None):
    """XQ [total_M, K] e4m3, WQ [G, N, K] e4m3, x_scale [total_M], w_scale [G, N] fp32,
    offsets [G] int32 inclusive prefix (group g owns rows [offsets[g-1], offsets[g]))
    -> out [total_M, N] bf16 (rows past offsets[G-1] zeroed when out is allocated here)."""
    import torch
    _check(XQ, "XQ", _fp8_types(), 2)
    _check(WQ, "WQ", _fp8_types(), 3)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    _check(offsets, "offsets", (torch.int32,), 1)
    total_M, K = XQ.shape
    G, N, K2 = WQ.shape
    if K2 != K or x_scale.numel() != total_M or w_scale.numel() != G * N or offsets.numel() != G:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.zeros((total_M, N), dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,), 2)
    s = mslkb_f8f8bf16_rowwise_grouped_offsets(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(),
        offsets.data_ptr(), out.data_ptr(), total_M, G, N, K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_rowwise_grouped_offsets")
    return out


def f8f8bf16_rowwise_grouped_batched(XQ, WQ, x_scale, w_scale, out=None, stream=None):
    """XQ [G, M, K] e4m3, WQ [G, N, K] e4m3, x_scale [G, M], w_scale [G, N] fp32
    -> out [G, M, N] bf16; every row of every slab computed."""
    import torch
    _check(XQ, "XQ", _fp8_types(), 3)
    _check(WQ, "WQ", _fp8_types(), 3)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    G, M, K = XQ.shape
    G2, N, K2 = WQ.shape
    if G2 != G or K2 != K or x_scale.numel() != G * M or w_scale.numel() != G * N:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((G, M, N), dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,))
    s = mslkb_f8f8bf16_rowwise_grouped_batched(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(), out.data_ptr(),
        G, M, N, K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_rowwise_grouped_batched")
    return out


def f8f8bf16_rowwise_grouped_n_offsets(XQ, WQ, x_scale, w_scale, offsets, out=None,
                                       stream=None):
    """Ragged N (3D-2D): XQ [G, M, K] e4m3, WQ [total_N, K] e4m3, x_scale [G, M] fp32,
    w_scale [total_N] fp32, offsets [G] int32 inclusive prefix over N -> out [M, total_N]
    bf16 (columns past offsets[G-1] zeroed when out is allocated here)."""
    import torch
    _check(XQ, "XQ", _fp8_types(), 3)
    _check(WQ, "WQ", _fp8_types(), 2)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    _check(offsets, "offsets", (torch.int32,), 1)
    G, M, K = XQ.shape
    total_N, K2 = WQ.shape
    if K2 != K or x_scale.numel() != G * M or w_scale.numel() != total_N or offsets.numel() != G:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.zeros((M, total_N), dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,), 2)
        if tuple(out.shape) != (M, total_N):
            raise ValueError("out has the wrong shape")
    s = mslkb_f8f8bf16_rowwise_grouped_n_offsets(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(),
        offsets.data_ptr(), out.data_ptr(), G, M, total_N, K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_rowwise_grouped_n_offsets")
    return out


def f8f8bf16_rowwise_grouped_k_offsets(XQ, WQ, x_scale, w_scale, offsets, out=None,
                                       stream=None):
    """Ragged K (2D-2D): XQ [M, total_K] e4m3, WQ [N, total_K] e4m3, x_scale [G, M] fp32,
    w_scale [G, N] fp32, offsets [G] int32 inclusive prefix over K -> out [G, M, N] bf16."""
    import torch
    _check(XQ, "XQ", _fp8_types(), 2)
    _check(WQ, "WQ", _fp8_types(), 2)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    _check(offsets, "offsets", (torch.int32,), 1)
    M, total_K = XQ.shape
    N, K2 = WQ.shape
    G = offsets.numel()
    if K2 != total_K or x_scale.numel() != G * M or w_scale.numel() != G * N:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((G, M, N), dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,))
        if out.numel() != G * M * N:
            raise ValueError("out has the wrong size")
    s = mslkb_f8f8bf16_rowwise_grouped_k_offsets(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(),
        offsets.data_ptr(), out.data_ptr(), G, M, N, total_K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_rowwise_grouped_k_offsets")
    return out


def f8f8bf16_groupwise_grouped_stacked(XQ, WQ, x_scale, w_scale, m_sizes, out=None,
                                       stream=None):
    """Block-scaled stacked: XQ [total_M, K] e4m3, WQ [G, N, K] e4m3, x_scale [total_M,
    K/128] fp32, w_scale [G, N/128, K/128] fp32, m_sizes [G] int64 -> out [total_M, N] bf16
    (K and N multiples of 128)."""
    import torch
    _check(XQ, "XQ", _fp8_types(), 2)
    _check(WQ, "WQ", _fp8_types(), 3)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    _check(m_sizes, "m_sizes", (torch.int64,), 1)
    total_M, K = XQ.shape
    G, N, K2 = WQ.shape
    if K2 != K or K % 128 or N % 128 or x_scale.numel() != total_M * (K // 128) \
            or w_scale.numel() != G * (N // 128) * (K // 128) or m_sizes.numel() != G:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.zeros((total_M, N), dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,), 2)
    s = mslkb_f8f8bf16_groupwise_grouped_stacked(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(),
        m_sizes.data_ptr(), out.data_ptr(), total_M, G, N, K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_groupwise_grouped_stacked")
    return out


def f8f8bf16_groupwise_grouped_dynamic(XQ, WQ, x_scale, w_scale, zero_start_index_M, out=None,
                                       stream=None):
    """Block-scaled dynamic: XQ [G, E, K] (or [G*E, K]) e4m3, WQ [G, N, K] e4m3, x_scale
    [G*E, K/128] fp32, w_scale [G, N/128, K/128] fp32, zero_start_index_M [G] int64
    -> out [G, E, N] (or [G*E, N]) bf16 with every padding row +0.0 (K, N multiples of
    128)."""
    import torch
    _check(XQ, "XQ", _fp8_types(), (2, 3))
    _check(WQ, "WQ", _fp8_types(), 3)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    _check(zero_start_index_M, "zero_start_index_M", (torch.int64,), 1)
    G, N, K = WQ.shape
    if XQ.dim() == 3:
        if XQ.shape[0] != G:
            raise ValueError("XQ and WQ disagree on G")
        E = XQ.shape[1]
        out_shape = (G, E, N)
    else:
        if G == 0 or XQ.shape[0] % G:
            raise ValueError("XQ rows must be G * expected_m")
        E = XQ.shape[0] // G
        out_shape = (G * E, N)
    if XQ.shape[-1] != K or K % 128 or N % 128 or x_scale.numel() != G * E * (K // 128) \
            or w_scale.numel() != G * (N // 128) * (K // 128) \
            or zero_start_index_M.numel() != G:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty(out_shape, dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,))
        if out.numel() != G * E * N:
            raise ValueError("out has the wrong size")
    s = mslkb_f8f8bf16_groupwise_grouped_dynamic(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(),
        zero_start_index_M.data_ptr(), out.data_ptr(), G, E, N, K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_groupwise_grouped_dynamic")
    return out


def f8f8bf16_groupwise_grouped_batched(XQ, WQ, x_scale, w_scale, out=None, stream=None):
    """Block-scaled batched: XQ [G, M, K] e4m3, WQ [G, N, K] e4m3, x_scale [G, M, K/128],
    w_scale [G, N/128, K/128] fp32 -> out [G, M, N] bf16; every slab row computed."""
    import torch
    _check(XQ, "XQ", _fp8_types(), 3)
    _check(WQ, "WQ", _fp8_types(), 3)
    _check(x_scale, "x_scale", (torch.float32,))
    _check(w_scale, "w_scale", (torch.float32,))
    G, M, K = XQ.shape
    G2, N, K2 = WQ.shape
    if G2 != G or K2 != K or K % 128 or N % 128 or x_scale.numel() != G * M * (K // 128) \
            or w_scale.numel() != G * (N // 128) * (K // 128):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((G, M, N), dtype=torch.bfloat16, device=XQ.device)
    else:
        _check(out, "out", (torch.bfloat16,))
        if out.numel() != G * M * N:
            raise ValueError("out has the wrong size")
    s = mslkb_f8f8bf16_groupwise_grouped_batched(
        XQ.data_ptr(), WQ.data_ptr(), x_scale.data_ptr(), w_scale.data_ptr(), out.data_ptr(),
        G, M, N, K, _stream_ptr(stream))
    if s != MSLKB_OK:
        raise MslkbError(s, "f8f8bf16_groupwise_grouped_batched")
    return out


def device_status(stream=None) -> int:
    """Read and clear the device status word (MSLKB_DEV_* bits)."""
    return mslkb_get_device_status(_stream_ptr(stream))
