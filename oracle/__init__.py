"""CPU oracle for the emulated FP8 scaled GEMM -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library under
``bit_exact_fp8_gb300``) never imports it and shares no code with it.

Two independent implementations live here:

* ``emu_oracle.c`` (loaded through ctypes): exact integer arithmetic, threaded
  over the host cores, fast enough for every workload (sampled at full size);
* ``spec.py``: a pure-Python model on ``fractions.Fraction`` for tiny cases,
  used to cross-check the C oracle.

Both follow the mmaemu v0.1 documentation pages ("User guide" section 1,
"Validation evidence" tables "Claims and their recordings", "Scope" and the
H100 PCIe probe table, "Limitations of mmaemu v0.1" section "Corrections of
earlier statements"); the readings taken where the pages are silent are listed
in the header of ``emu_oracle.c``.

Parity: pinned -- see tests/test_oracle_pins.py for what each part is pinned to.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "emu_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

FORMATS = {"e4m3fn": 0, "e5m2": 1}
OUT_DTYPES = {"f32": 0, "bf16": 1, "f16": 2, "e4m3fn": 3, "e5m2": 4}
OUT_NP = {"f32": np.uint32, "bf16": np.uint16, "f16": np.uint16, "e4m3fn": np.uint8,
          "e5m2": np.uint8}

#: instruction/platform presets: block width B, retained fraction bits F, slow
#: restart R, c in alignment, split scheme (0 contiguous, 1 interleaved),
#: k-tile of the split rule, combine (0 serial, 1 pairwise).
PRESETS = {
    # "Validation evidence", H100 PCIe probe table: 32-product blocks, 13 fraction
    # bits, c in the block's alignment, restart every 128, contiguous 128-wide
    # k-tiles combined serially.
    "hopper": dict(block_width=32, frac_bits=13, restart=128, c_in_alignment=1,
                   split_scheme=0, ktile=128, combine=0),
    # "Validation evidence", table "Claims and their recordings": 16-term blocks,
    # 13 fraction bits, an all-zero block still truncates c; 64-wide k-tiles dealt
    # round-robin; serial (or pairwise) combination.
    "ada": dict(block_width=16, frac_bits=13, restart=128, c_in_alignment=1,
                split_scheme=1, ktile=64, combine=0),
}


class Preset(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in
                ("block_width", "frac_bits", "restart", "c_in_alignment",
                 "split_scheme", "ktile", "combine")]


def build(force: bool = False) -> str:
    """Compile ``emu_oracle.c`` into ``liboracle.so`` (plain gcc, no GPU)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
                           _SRC, "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None

#: tests may point the wrapper at another build of emu_oracle.c (a mutant copy)
_LIB_OVERRIDE = os.environ.get("EMU_ORACLE_LIB")


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if _LIB_OVERRIDE:
            L = ctypes.CDLL(_LIB_OVERRIDE)
        else:
            build()
            L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
        L.oracle_scaled_mm.argtypes = [P, ctypes.c_int, P, ctypes.c_int, i64, i64, i64, u32, u32,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(Preset), P, ctypes.c_int, ctypes.c_int, u32]
        L.oracle_acc_sampled.argtypes = [P, ctypes.c_int, P, ctypes.c_int, i64, i64, i64,
                                         ctypes.c_int, ctypes.c_int, ctypes.POINTER(Preset),
                                         i64, P, P, P, ctypes.c_int]
        L.oracle_epilogue.argtypes = [P, i64, u32, u32, ctypes.c_int, P, ctypes.c_int, u32]
        L.oracle_f32_to_fp8.argtypes = [i64, P, ctypes.c_int, P]
        L.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_int, P]
        L.oracle_products.argtypes = [i64, P, ctypes.c_int, P, ctypes.c_int, P]
        L.oracle_blk_many.argtypes = [i64, P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int,
                                      ctypes.c_int, P]
        L.oracle_blk_exact.argtypes = [u32, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int,
                                       ctypes.c_int, P, P, P]
        for name in ("oracle_f32_add_rn", "oracle_f32_mul_rn", "oracle_f32_fma_plus0"):
            getattr(L, name).argtypes = [i64, P, P, P]
        L.oracle_f32_to_bf16.argtypes = [i64, P, P]
        L.oracle_f32_to_f16.argtypes = [i64, P, P]
        L.oracle_split_indices.argtypes = [i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, P]
        L.oracle_split_indices.restype = i64
        L.oracle_combine.argtypes = [P, ctypes.c_int, ctypes.c_int]
        L.oracle_combine.restype = u32
        L.oracle_chain.argtypes = [i64, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
        L.oracle_round.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int]
        L.oracle_round.restype = u32
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _preset(preset) -> Preset:
    if isinstance(preset, str):
        preset = PRESETS[preset]
    return Preset(**preset)


def _f32_bits(x) -> int:
    return int(np.array(x, dtype=np.float32).view(np.uint32))


def _check(st: int, what: str):
    if st != 0:
        raise RuntimeError(f"oracle {what} failed with status {st}")


def scaled_mm(a_codes: np.ndarray, b_codes_nk: np.ndarray, fmt_a: str, fmt_b: str,
              scale_a: float, scale_b: float, out_dtype: str = "bf16",
              fast_accum: bool = True, split_S: int = 1, preset="hopper",
              nthreads: int = 0, scale_result=None) -> np.ndarray:
    """Full GEMM.  ``a_codes`` [M,K] uint8 (row-major), ``b_codes_nk`` [N,K] uint8:
    the bytes of mat2 [K,N] column-major.  Returns the output bit patterns
    [M,N] (uint32 for f32, uint16 for bf16/f16)."""
    a = np.ascontiguousarray(a_codes, dtype=np.uint8)
    b = np.ascontiguousarray(b_codes_nk, dtype=np.uint8)
    M, K = a.shape
    N, K2 = b.shape
    assert K == K2
    out = np.zeros((M, N), dtype=OUT_NP[out_dtype])
    p = _preset(preset)
    st = lib().oracle_scaled_mm(_ptr(a), FORMATS[fmt_a], _ptr(b), FORMATS[fmt_b], M, N, K,
                                _f32_bits(scale_a), _f32_bits(scale_b), OUT_DTYPES[out_dtype],
                                int(bool(fast_accum)), int(split_S), ctypes.byref(p), _ptr(out),
                                int(nthreads), int(scale_result is not None),
                                _f32_bits(1.0 if scale_result is None else scale_result))
    _check(st, "scaled_mm")
    return out


def acc_sampled(a_codes: np.ndarray, b_codes_nk: np.ndarray, fmt_a: str, fmt_b: str,
                idx_m: np.ndarray, idx_n: np.ndarray, fast_accum: bool = True,
                split_S: int = 1, preset="hopper", nthreads: int = 0) -> np.ndarray:
    """fp32 accumulator bits (before the scales) at the outputs (idx_m[i], idx_n[i])."""
    a = np.ascontiguousarray(a_codes, dtype=np.uint8)
    b = np.ascontiguousarray(b_codes_nk, dtype=np.uint8)
    M, K = a.shape
    N, _ = b.shape
    im = np.ascontiguousarray(idx_m, dtype=np.int64)
    jn = np.ascontiguousarray(idx_n, dtype=np.int64)
    out = np.zeros(im.shape[0], dtype=np.uint32)
    p = _preset(preset)
    st = lib().oracle_acc_sampled(_ptr(a), FORMATS[fmt_a], _ptr(b), FORMATS[fmt_b], M, N, K,
                                  int(bool(fast_accum)), int(split_S), ctypes.byref(p),
                                  im.shape[0], _ptr(im), _ptr(jn), _ptr(out), int(nthreads))
    _check(st, "acc_sampled")
    return out


def epilogue(acc_bits: np.ndarray, scale_a: float, scale_b: float, out_dtype: str,
             scale_result=None) -> np.ndarray:
    acc = np.ascontiguousarray(acc_bits, dtype=np.uint32)
    out = np.zeros(acc.shape, dtype=OUT_NP[out_dtype])
    st = lib().oracle_epilogue(_ptr(acc), acc.size, _f32_bits(scale_a), _f32_bits(scale_b),
                               OUT_DTYPES[out_dtype], _ptr(out), int(scale_result is not None),
                               _f32_bits(1.0 if scale_result is None else scale_result))
    _check(st, "epilogue")
    return out


def decode(fmt: str, code: int):
    """(nan, inf, neg, sig, e, f): value = (-1)^neg * sig * 2^(e - f)."""
    out = np.zeros(6, dtype=np.int32)
    _check(lib().oracle_decode(FORMATS[fmt], int(code), _ptr(out)), "decode")
    return tuple(int(v) for v in out)


def products(a: np.ndarray, fmt_a: str, b: np.ndarray, fmt_b: str) -> np.ndarray:
    """[n,4] int32 rows (neg, sig, e, f) of the exact products a[i] x b[i]."""
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.zeros((a.size, 4), dtype=np.int32)
    lib().oracle_products(a.size, _ptr(a), FORMATS[fmt_a], _ptr(b), FORMATS[fmt_b], _ptr(out))
    return out


def blk_many(c_bits: np.ndarray, a: np.ndarray, fmt_a: str, b: np.ndarray, fmt_b: str,
             F: int = 13) -> np.ndarray:
    """Block results for ``count`` independent blocks: ``a``/``b`` are [count, n]."""
    c = np.ascontiguousarray(c_bits, dtype=np.uint32)
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    count, n = a.shape
    out = np.zeros(count, dtype=np.uint32)
    _check(lib().oracle_blk_many(count, _ptr(c), n, _ptr(a), FORMATS[fmt_a], _ptr(b),
                                 FORMATS[fmt_b], F, _ptr(out)), "blk_many")
    return out


def blk_exact(c_bits: int, a: np.ndarray, fmt_a: str, b: np.ndarray, fmt_b: str, F: int):
    """(nonzero, S, E): the exact block sum S in units of 2^(E-F)."""
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    hi = np.zeros(1, dtype=np.int64)
    lo = np.zeros(1, dtype=np.uint64)
    E = np.zeros(1, dtype=np.int32)
    r = lib().oracle_blk_exact(int(c_bits), a.size, _ptr(a), FORMATS[fmt_a], _ptr(b),
                               FORMATS[fmt_b], int(F), _ptr(hi), _ptr(lo), _ptr(E))
    if r < 0:
        raise RuntimeError(f"oracle blk_exact status {r}")
    S = (int(hi[0]) << 64) | int(lo[0])
    return bool(r), S, int(E[0])


def _vec2(name, a, b):
    a = np.ascontiguousarray(a, dtype=np.uint32)
    b = np.ascontiguousarray(b, dtype=np.uint32)
    out = np.zeros(a.shape, dtype=np.uint32)
    getattr(lib(), name)(a.size, _ptr(a), _ptr(b), _ptr(out))
    return out


def f32_add_rn(a_bits, b_bits):
    return _vec2("oracle_f32_add_rn", a_bits, b_bits)


def f32_mul_rn(a_bits, b_bits):
    return _vec2("oracle_f32_mul_rn", a_bits, b_bits)


def f32_fma_plus0(a_bits, b_bits):
    return _vec2("oracle_f32_fma_plus0", a_bits, b_bits)


def f32_to_bf16(a_bits):
    a = np.ascontiguousarray(a_bits, dtype=np.uint32)
    out = np.zeros(a.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16(a.size, _ptr(a), _ptr(out))
    return out


def f32_to_f16(a_bits):
    a = np.ascontiguousarray(a_bits, dtype=np.uint32)
    out = np.zeros(a.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16(a.size, _ptr(a), _ptr(out))
    return out


def f32_to_fp8(a_bits, fmt: str) -> np.ndarray:
    """fp32 -> FP8 codes, round to nearest even, saturating (NaN -> 0x7F)."""
    a = np.ascontiguousarray(a_bits, dtype=np.uint32)
    out = np.zeros(a.shape, dtype=np.uint8)
    _check(lib().oracle_f32_to_fp8(a.size, _ptr(a), FORMATS[fmt], _ptr(out)), "f32_to_fp8")
    return out


def split_indices(K: int, S: int, scheme: int, ktile: int, s: int) -> np.ndarray:
    idx = np.zeros(max(K, 1), dtype=np.int64)
    n = lib().oracle_split_indices(K, S, scheme, ktile, s, _ptr(idx))
    if n < 0:
        raise ValueError("bad split arguments")
    return idx[:n].copy()


def combine(partials_bits, pairwise: bool) -> int:
    p = np.ascontiguousarray(partials_bits, dtype=np.uint32)
    return int(lib().oracle_combine(_ptr(p), p.size, int(bool(pairwise))))


def chain(a: np.ndarray, fmt_a: str, b: np.ndarray, fmt_b: str, fast: bool,
          B: int = 32, F: int = 13, R: int = 128) -> int:
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.zeros(1, dtype=np.uint32)
    _check(lib().oracle_chain(a.size, _ptr(a), FORMATS[fmt_a], _ptr(b), FORMATS[fmt_b],
                              int(bool(fast)), B, F, R, _ptr(out)), "chain")
    return int(out[0])


def round_bits(neg: int, mag: int, exp2: int, fmt: int = 0, mode: int = 0) -> int:
    """Round (-1)^neg * mag * 2^exp2 into fp32 (fmt 0), bf16 (1), fp16 (2);
    mode 0 nearest-even, 1 toward zero."""
    return int(lib().oracle_round(int(neg), (mag >> 64) & (2**64 - 1), mag & (2**64 - 1),
                                  int(exp2), int(fmt), int(mode)))
