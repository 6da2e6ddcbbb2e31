"""ctypes binding of libemufp8 (include/emu_fp8.h): the C entry points under the
same names, argument marshalling only.  Every step of the GEMM runs in the
library's CUDA kernels; there is no Python or CPU fallback.  If the library is
missing, every call raises."""
from __future__ import annotations

import ctypes
import os

from .build import LIB

EMU_OK = 0
EMU_EINVAL = -1
EMU_EREJECT = -2
EMU_EUNSUPPORTED = -3
EMU_ECUDA = -4

EMU_E4M3FN = 0
EMU_E5M2 = 1
EMU_OUT_F32 = 0
EMU_OUT_BF16 = 1
EMU_OUT_F16 = 2
EMU_OUT_E4M3FN = 3
EMU_OUT_E5M2 = 4

#: every symbol include/emu_fp8.h declares
EXPORTED = ("emu_preset_get", "emu_workspace_bytes", "emu_scaled_mm", "emu_last_error",
            "emu_abi_version", "emu_scaled_mm_noalloc", "emu_device_status",
            "emu_selftest_wait_timeout", "emu_scaled_mm_ex", "emu_host_staging_bytes",
            "emu_scaled_mm_host", "emu_tile_for", "emu_tc_selftest")

#: size of the static scratch of emu_scaled_mm_noalloc (EMU_NOALLOC_SCRATCH_BYTES)
EMU_NOALLOC_SCRATCH_BYTES = 4 << 20


class emu_preset_t(ctypes.Structure):
    _fields_ = [("block_width", ctypes.c_int32), ("frac_bits", ctypes.c_int32),
                ("restart", ctypes.c_int32), ("c_in_alignment", ctypes.c_int32),
                ("split_scheme", ctypes.c_int32), ("ktile", ctypes.c_int32),
                ("combine", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_handle = None


def load(path: str = LIB) -> ctypes.CDLL:
    """Load libemufp8.so (raises OSError if it has not been built)."""
    global _handle
    if _handle is not None:
        return _handle
    if not os.path.exists(path):
        raise OSError(f"libemufp8 is not built ({path} missing): run "
                      "python -m bit_exact_fp8_gb300.build")
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    L.emu_preset_get.argtypes = [ctypes.c_char_p, ctypes.POINTER(emu_preset_t)]
    L.emu_preset_get.restype = ctypes.c_int
    L.emu_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]
    L.emu_workspace_bytes.restype = ctypes.c_size_t
    L.emu_scaled_mm.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_int64, P, P, P, ctypes.c_int, ctypes.c_int32,
                                ctypes.c_int32, ctypes.POINTER(emu_preset_t), P, ctypes.c_size_t, P]
    L.emu_scaled_mm.restype = ctypes.c_int
    L.emu_scaled_mm_ex.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_int64, P, P, P, P, ctypes.c_int,
                                   ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(emu_preset_t),
                                   P, ctypes.c_size_t, P]
    L.emu_scaled_mm_ex.restype = ctypes.c_int
    L.emu_scaled_mm_noalloc.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, P, P, P, ctypes.c_int,
                                        ctypes.c_int32, ctypes.c_int32,
                                        ctypes.POINTER(emu_preset_t), P]
    L.emu_scaled_mm_noalloc.restype = ctypes.c_int
    L.emu_host_staging_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int32, ctypes.c_int]
    L.emu_host_staging_bytes.restype = ctypes.c_size_t
    L.emu_scaled_mm_host.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                     ctypes.c_float, P, P, ctypes.c_int, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.POINTER(emu_preset_t), P,
                                     ctypes.c_size_t, ctypes.c_int32, P]
    L.emu_scaled_mm_host.restype = ctypes.c_int
    L.emu_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int32]
    L.emu_device_status.restype = ctypes.c_int
    L.emu_tc_selftest.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.emu_tc_selftest.restype = ctypes.c_int
    L.emu_selftest_wait_timeout.argtypes = [P]
    L.emu_selftest_wait_timeout.restype = ctypes.c_int
    L.emu_tile_for.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                               ctypes.c_int32, ctypes.POINTER(emu_preset_t), ctypes.c_int32,
                               ctypes.c_char_p, ctypes.c_size_t]
    L.emu_tile_for.restype = ctypes.c_int
    L.emu_last_error.argtypes = []
    L.emu_last_error.restype = ctypes.c_char_p
    L.emu_abi_version.argtypes = []
    L.emu_abi_version.restype = ctypes.c_int
    _handle = L
    return L


def emu_preset_get(name: str) -> emu_preset_t:
    p = emu_preset_t()
    st = load().emu_preset_get(name.encode(), ctypes.byref(p))
    if st != EMU_OK:
        raise KeyError(f"unknown preset {name!r}")
    return p


def emu_workspace_bytes(M: int, N: int, split_S: int) -> int:
    return int(load().emu_workspace_bytes(M, N, split_S))


def emu_last_error() -> str:
    return load().emu_last_error().decode(errors="replace")


def emu_abi_version() -> int:
    return int(load().emu_abi_version())


def emu_scaled_mm(A: int, fmt_a: int, B: int, fmt_b: int, M: int, N: int, K: int,
                  scale_a: int, scale_b: int, out: int, out_dtype: int, fast_accum: int,
                  split_S: int, preset: emu_preset_t, workspace: int, workspace_bytes: int,
                  stream: int) -> int:
    """The C call with raw device addresses (ints); returns the status code."""
    return int(load().emu_scaled_mm(
        ctypes.c_void_p(A), fmt_a, ctypes.c_void_p(B), fmt_b, M, N, K,
        ctypes.c_void_p(scale_a), ctypes.c_void_p(scale_b), ctypes.c_void_p(out), out_dtype,
        int(fast_accum), int(split_S), ctypes.byref(preset), ctypes.c_void_p(workspace),
        int(workspace_bytes), ctypes.c_void_p(stream)))


def emu_scaled_mm_noalloc(A: int, fmt_a: int, B: int, fmt_b: int, M: int, N: int, K: int,
                          scale_a: int, scale_b: int, out: int, out_dtype: int, fast_accum: int,
                          split_S: int, preset: emu_preset_t, stream: int) -> int:
    """The C call that keeps split partials in the library's static device scratch
    (for callers that cannot allocate a workspace); returns the status code."""
    return int(load().emu_scaled_mm_noalloc(
        ctypes.c_void_p(A), fmt_a, ctypes.c_void_p(B), fmt_b, M, N, K,
        ctypes.c_void_p(scale_a), ctypes.c_void_p(scale_b), ctypes.c_void_p(out), out_dtype,
        int(fast_accum), int(split_S), ctypes.byref(preset), ctypes.c_void_p(stream)))


def emu_host_staging_bytes(M: int, N: int, K: int, split_S: int, out_dtype: int) -> int:
    return int(load().emu_host_staging_bytes(M, N, K, split_S, out_dtype))


def emu_scaled_mm_host(A_host: int, fmt_a: int, B_host: int, fmt_b: int, M: int, N: int, K: int,
                       scale_a: float, scale_b: float, scale_result, out_host: int,
                       out_dtype: int, fast_accum: int, split_S: int, preset: emu_preset_t,
                       staging: int, staging_bytes: int, chunks: int, stream: int) -> int:
    """The C call with host operand/result addresses and a device staging buffer
    (ints); scale_result is None or a float (passed by host pointer).  Asynchronous:
    the result is in out_host once `stream` completes.  Returns the status code."""
    sr = None if scale_result is None else ctypes.c_float(float(scale_result))
    return int(load().emu_scaled_mm_host(
        ctypes.c_void_p(A_host), fmt_a, ctypes.c_void_p(B_host), fmt_b, M, N, K,
        float(scale_a), float(scale_b), None if sr is None else ctypes.byref(sr),
        ctypes.c_void_p(out_host), out_dtype, int(fast_accum), int(split_S),
        ctypes.byref(preset), ctypes.c_void_p(staging), int(staging_bytes), int(chunks),
        ctypes.c_void_p(stream)))


def emu_device_status(reset: bool = False) -> int:
    """The library's device status word (0 ok, 1 a bounded wait gave up); synchronous."""
    v = ctypes.c_int32(0)
    st = load().emu_device_status(ctypes.byref(v), int(bool(reset)))
    if st != EMU_OK:
        raise RuntimeError(f"emu_device_status failed: {emu_last_error()}")
    return int(v.value)


def emu_tc_selftest() -> int:
    """Outputs of the tensor-core product self-test that differ from the exact product
    (0: exact), 0xFFFFFFFF if a wait gave up; raises on a CUDA error."""
    v = ctypes.c_uint32(0)
    st = load().emu_tc_selftest(ctypes.byref(v))
    if st != EMU_OK:
        raise RuntimeError(f"emu_tc_selftest failed: {emu_last_error()}")
    return int(v.value)


def emu_selftest_wait_timeout(stream: int = 0) -> int:
    return int(load().emu_selftest_wait_timeout(ctypes.c_void_p(stream)))


def emu_tile_for(M: int, N: int, K: int, fast_accum: int, split_S: int, preset: emu_preset_t,
                 sm_count: int = 0) -> "tuple[int, str]":
    """(status, tile name) of emu_tile_for."""
    buf = ctypes.create_string_buffer(16)
    st = load().emu_tile_for(M, N, K, int(fast_accum), int(split_S), ctypes.byref(preset),
                             int(sm_count), buf, len(buf))
    return int(st), buf.value.decode()


def emu_scaled_mm_ex(A: int, fmt_a: int, B: int, fmt_b: int, M: int, N: int, K: int,
                     scale_a: int, scale_b: int, scale_result: int, out: int, out_dtype: int,
                     fast_accum: int, split_S: int, preset: emu_preset_t, workspace: int,
                     workspace_bytes: int, stream: int) -> int:
    """emu_scaled_mm with scale_result (0: none) for FP8 outputs; returns the status."""
    return int(load().emu_scaled_mm_ex(
        ctypes.c_void_p(A), fmt_a, ctypes.c_void_p(B), fmt_b, M, N, K,
        ctypes.c_void_p(scale_a), ctypes.c_void_p(scale_b), ctypes.c_void_p(scale_result or None),
        ctypes.c_void_p(out), out_dtype, int(fast_accum), int(split_S), ctypes.byref(preset),
        ctypes.c_void_p(workspace), int(workspace_bytes), ctypes.c_void_p(stream)))
