"""ctypes binding of libemupeaks: the measured instruction rates of the GB300 pipes
that the emulated GEMM issues on (lane-operations per clock per SM), which
bench.py takes as its roofline denominators, and the check that packed f32x2
arithmetic rounds each half exactly as the scalar instruction does."""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Tuple

from .build import PEAKS_LIB

_handle = None


def load(path: str = PEAKS_LIB) -> ctypes.CDLL:
    global _handle
    if _handle is not None:
        return _handle
    if not os.path.exists(path):
        raise OSError(f"libemupeaks is not built ({path} missing): run "
                      "python -m bit_exact_fp8_gb300.build")
    L = ctypes.CDLL(path)
    L.emu_peaks_count.restype = ctypes.c_int
    L.emu_peaks_name.argtypes = [ctypes.c_int]
    L.emu_peaks_name.restype = ctypes.c_char_p
    L.emu_peaks_measure.argtypes = [ctypes.POINTER(ctypes.c_double)]
    L.emu_peaks_measure.restype = ctypes.c_int
    L.emu_peaks_f32x2_agreement.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint)]
    L.emu_peaks_f32x2_agreement.restype = ctypes.c_int
    _handle = L
    return L


def issue_rates() -> Dict[str, float]:
    """Lane-operations per clock per SM of each measured operation on the current
    CUDA device (``emulation_mix_macs``: MACs per clock per SM of the GEMM's
    arithmetic mix of 1.5 packed FP32 instructions and 0.5 DPX per MAC)."""
    L = load()
    n = L.emu_peaks_count()
    buf = (ctypes.c_double * n)()
    st = L.emu_peaks_measure(buf)
    if st != 0:
        raise RuntimeError(f"emu_peaks_measure failed ({st})")
    return {L.emu_peaks_name(i).decode(): float(buf[i]) for i in range(n)}


def f32x2_agreement(n: int = 1 << 22) -> Tuple[int, int, int]:
    """Halves of n random operand pairs where mul.rn / mul.rz / add.rn .f32x2 differ
    from the scalar instruction (subnormal results included)."""
    L = load()
    bad = (ctypes.c_uint * 3)()
    st = L.emu_peaks_f32x2_agreement(n, bad)
    if st != 0:
        raise RuntimeError(f"emu_peaks_f32x2_agreement failed ({st})")
    return int(bad[0]), int(bad[1]), int(bad[2])
