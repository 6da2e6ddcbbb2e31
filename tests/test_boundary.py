"""CPU tests of the C ABI: the library loads, exports every symbol include/*.h
declares, and its host-side checks return the documented status before any
launch (no GPU is touched: every call here fails its argument checks first)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_exact_fp8_gb300 import _lib, build
    build.build()
    return _lib


def declared_functions(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(emu_\w+)\s*\(", src, flags=re.M))


def test_headers_are_the_two_libraries():
    assert sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")) == \
        ["emu_fp8.h", "emu_peaks.h"]


def test_library_exports_every_declared_symbol(lib):
    L = lib.load()
    declared = declared_functions("emu_fp8.h")
    assert {"emu_scaled_mm", "emu_workspace_bytes", "emu_preset_get"} <= declared
    for name in declared:
        assert hasattr(L, name), name
    assert set(lib.EXPORTED) == declared


def test_peaks_library_exports_every_declared_symbol(lib):
    from bit_exact_fp8_gb300 import peaks
    L = peaks.load()
    declared = declared_functions("emu_peaks.h")
    assert declared == {"emu_peaks_count", "emu_peaks_name", "emu_peaks_measure",
                        "emu_peaks_f32x2_agreement"}
    for name in declared:
        assert hasattr(L, name), name
    assert L.emu_peaks_count() == 17
    assert L.emu_peaks_name(12) == b"emulation_mix_macs"
    assert L.emu_peaks_name(15) == b"emulation_mix_vector_macs"
    assert L.emu_peaks_name(16) == b"emulation_tile_macs" and L.emu_peaks_name(17) == b""


def test_presets_and_abi(lib):
    assert lib.emu_abi_version() == 1
    h = lib.emu_preset_get("hopper").as_dict()
    assert h == dict(block_width=32, frac_bits=13, restart=128, c_in_alignment=1,
                     split_scheme=0, ktile=128, combine=0)
    a = lib.emu_preset_get("ada").as_dict()
    assert a == dict(block_width=16, frac_bits=13, restart=128, c_in_alignment=1,
                     split_scheme=1, ktile=64, combine=0)
    with pytest.raises(KeyError):
        lib.emu_preset_get("sm_120")
    import oracle
    assert oracle.PRESETS["hopper"] == h and oracle.PRESETS["ada"] == a


def test_workspace_bytes(lib):
    assert lib.emu_workspace_bytes(16, 256, 1) == 0
    assert lib.emu_workspace_bytes(16, 256, 24) == 24 * 16 * 256 * 4
    assert lib.emu_workspace_bytes(3, 16, 2) == 512          # rounded up to 256
    assert lib.emu_workspace_bytes(-1, 16, 2) == 0


FAKE = 1 << 20   # a 16-byte aligned non-null address; never dereferenced here


def call(lib, **kw):
    args = dict(A=FAKE, fmt_a=0, B=FAKE, fmt_b=0, M=16, N=64, K=256, scale_a=FAKE,
                scale_b=FAKE, out=FAKE, out_dtype=1, fast_accum=1, split_S=1,
                preset=lib.emu_preset_get("hopper"), workspace=0, workspace_bytes=0, stream=0)
    args.update(kw)
    return lib.emu_scaled_mm(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt_a=1, fmt_b=1), -2),                 # e5m2 x e5m2 rejected by torch
    (dict(K=250), -2),                            # K not a multiple of 16
    (dict(N=72), -2),                             # N not a multiple of 16
    (dict(A=FAKE + 8), -2),                       # misaligned storage
    (dict(out=FAKE + 4), -2),
    (dict(fmt_a=2), -1),
    (dict(out_dtype=5), -1),
    (dict(M=-1), -1),
    (dict(split_S=0), -1),
    (dict(split_S=65), -3),
    (dict(split_S=2), -1),                        # workspace missing
    (dict(split_S=2, workspace=FAKE, workspace_bytes=100), -1),
    (dict(scale_a=0), -1),
    (dict(A=0), -1),
    (dict(K=1 << 31), -3),
])
def test_argument_errors(lib, kw, status):
    st = call(lib, **kw)
    assert st == status, lib.emu_last_error()
    assert lib.emu_last_error() != ""


@pytest.mark.parametrize("field,value,status", [
    ("block_width", 8, -3), ("frac_bits", 12, -3), ("c_in_alignment", 0, -3),
    ("restart", 40, -3), ("ktile", 48, -3), ("split_scheme", 2, -1), ("combine", 2, -1)])
def test_preset_errors(lib, field, value, status):
    p = lib.emu_preset_get("hopper")
    setattr(p, field, value)
    assert call(lib, preset=p) == status


def test_null_preset(lib):
    L = lib.load()
    st = L.emu_scaled_mm(None, 0, None, 0, 1, 16, 16, None, None, None, 0, 1, 1, None, None, 0, None)
    assert st == -1


def test_zero_sized_is_noop(lib):
    # M == 0 or N == 0: success, nothing enqueued (no pointer needed)
    assert call(lib, M=0, A=0, B=0, out=0, scale_a=0, scale_b=0) == 0
    assert call(lib, N=0, A=0, B=0, out=0, scale_a=0, scale_b=0) == 0


def test_python_api_rejects_cpu_and_unsupported():
    from bit_exact_fp8_gb300 import (ReferenceRejectsError, UnsupportedFeatureError,
                                     scaled_mm)
    x = torch.zeros(16, 32).to(torch.float8_e4m3fn)
    w = torch.zeros(16, 32).to(torch.float8_e4m3fn)
    one = torch.ones(())
    with pytest.raises(UnsupportedFeatureError):
        scaled_mm(x, w.t(), one, one, bias=torch.zeros(16))
    with pytest.raises(ValueError):                  # scale_result must live on the GPU
        scaled_mm(x, w.t(), one, one, scale_result=one)
    with pytest.raises(ReferenceRejectsError):
        scaled_mm(x.float(), w.t(), one, one)
    with pytest.raises(ValueError):                  # no CPU path
        scaled_mm(x, w.t(), one, one)
    assert issubclass(ReferenceRejectsError, RuntimeError)
    assert issubclass(UnsupportedFeatureError, NotImplementedError)


def test_fp8_output_argument_checks(lib):
    L = lib.load()
    p = lib.emu_preset_get("hopper")
    def ex(fa, fb, od, sr):
        return lib.emu_scaled_mm_ex(FAKE, fa, FAKE, fb, 16, 64, 256, FAKE, FAKE, sr, FAKE, od,
                                    1, 1, p, 0, 0, 0)
    assert ex(0, 0, 4, 0) == -2          # cuBLASLt refuses e4m3 x e4m3 -> e5m2
    assert ex(0, 0, 1, FAKE) == -3       # scale_result with a non-fp8 output
    assert ex(0, 0, 5, 0) == -1          # unknown output dtype
    assert L is not None


def test_host_staging_bytes(lib):
    # scalars (256) | A | B | out | partials, each rounded up to 256 bytes
    r = lambda x: (x + 255) // 256 * 256
    M, N, K = 64, 5760, 1920
    assert lib.emu_host_staging_bytes(M, N, K, 1, lib.EMU_OUT_BF16) == \
        256 + r(M * K) + r(N * K) + r(M * N * 2)
    assert lib.emu_host_staging_bytes(16, 256, 4096, 8, lib.EMU_OUT_F32) == \
        256 + r(16 * 4096) + r(256 * 4096) + r(16 * 256 * 4) + r(8 * 16 * 256 * 4)
    assert lib.emu_host_staging_bytes(3, 16, 32, 1, lib.EMU_OUT_E4M3FN) == 256 + 256 + 512 + 256
    assert lib.emu_host_staging_bytes(-1, 16, 32, 1, 0) == 0
    assert lib.emu_host_staging_bytes(1, 16, 32, 0, 0) == 0
    assert lib.emu_host_staging_bytes(1, 16, 32, 1, 5) == 0


def test_host_entry_point_argument_errors(lib):
    # every case fails its checks before any CUDA call (no GPU here)
    p = lib.emu_preset_get("hopper")
    need = lib.emu_host_staging_bytes(16, 64, 256, 1, lib.EMU_OUT_BF16)

    def host(**kw):
        a = dict(A=FAKE, fa=0, B=FAKE, fb=0, M=16, N=64, K=256, sa=1.0, sb=1.0, sr=None,
                 out=FAKE, od=lib.EMU_OUT_BF16, fast=1, S=1, staging=1 << 20,
                 staging_bytes=need, chunks=4)
        a.update(kw)
        return lib.emu_scaled_mm_host(a["A"], a["fa"], a["B"], a["fb"], a["M"], a["N"], a["K"],
                                      a["sa"], a["sb"], a["sr"], a["out"], a["od"], a["fast"],
                                      a["S"], p, a["staging"], a["staging_bytes"], a["chunks"], 0)
    assert host(fa=1, fb=1) == lib.EMU_EREJECT                  # e5m2 x e5m2
    assert host(od=lib.EMU_OUT_E5M2) == lib.EMU_EREJECT         # e4m3 x e4m3 -> e5m2
    assert host(sr=2.0) == lib.EMU_EUNSUPPORTED                 # scale_result, bf16 out
    assert host(N=40) == lib.EMU_EREJECT                        # N not a multiple of 16
    assert host(S=0) == lib.EMU_EINVAL
    assert host(out=0) == lib.EMU_EINVAL                        # null out_host
    assert host(A=0) == lib.EMU_EINVAL                          # null operand
    assert host(staging_bytes=need - 1) == lib.EMU_EINVAL       # short staging
    assert "staging" in lib.emu_last_error()
    assert host(staging=(1 << 20) + 16) == lib.EMU_EINVAL       # not 256-byte aligned
    assert host(M=0, A=0, B=0, out=0, staging=0, staging_bytes=0) == lib.EMU_OK   # no-op


def test_python_host_api_rejects_device_and_bad_dtypes():
    from bit_exact_fp8_gb300 import ReferenceRejectsError, scaled_mm_host
    x = torch.zeros(16, 32).to(torch.float8_e4m3fn)
    w = torch.zeros(16, 32).to(torch.float8_e4m3fn)
    with pytest.raises(ReferenceRejectsError):
        scaled_mm_host(x.float(), w.t(), 1.0, 1.0)
    with pytest.raises(ValueError):
        scaled_mm_host(x, w, 1.0, 1.0)                          # [16,32] @ [16,32]


def test_workspace_bytes_never_wraps(lib):
    # S * M * N * 4 beyond size_t: SIZE_MAX, so no workspace passes the size check
    big = (1 << 31) - 1
    assert lib.emu_workspace_bytes(big, big, 64) == (1 << 64) - 1
    assert lib.emu_workspace_bytes(1 << 30, 1 << 30, 64) == (1 << 64) - 1
    assert lib.emu_workspace_bytes(1 << 20, 1 << 20, 64) == 64 * (1 << 40) * 4
    assert lib.emu_workspace_bytes(0, 1 << 30, 64) == 0
    st = call(lib, M=big, N=big - 15, split_S=64, workspace=FAKE, workspace_bytes=1 << 40)
    assert st == -1 and "workspace" in lib.emu_last_error()


def _noalloc(lib, **kw):
    args = dict(A=FAKE, fmt_a=0, B=FAKE, fmt_b=0, M=16, N=64, K=256, scale_a=FAKE,
                scale_b=FAKE, out=FAKE, out_dtype=1, fast_accum=1, split_S=2,
                preset=lib.emu_preset_get("hopper"), stream=0)
    args.update(kw)
    return lib.emu_scaled_mm_noalloc(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt_a=1, fmt_b=1), -2),                 # e5m2 x e5m2: EREJECT, as emu_scaled_mm
    (dict(K=250), -2),                            # K not a multiple of 16
    (dict(fmt_a=2), -1),                          # unknown format
    (dict(split_S=0), -1),
])
def test_noalloc_argument_statuses_come_before_the_scratch_limit(lib, kw, status):
    # the same statuses as emu_scaled_mm, even when the partials would not fit the
    # static scratch (S * M * N far above EMU_NOALLOC_SCRATCH_BYTES / 4)
    assert _noalloc(lib, M=1 << 20, N=1 << 20, **kw) == status
    assert _noalloc(lib, **kw) == status


def test_noalloc_scratch_limit_is_exact(lib):
    # one 16-column step above S * M * N = EMU_NOALLOC_SCRATCH_BYTES / 4 is refused on
    # the host (nothing touches a GPU); the exact fill itself runs in the GPU test
    limit = lib.EMU_NOALLOC_SCRATCH_BYTES // 4
    S, M = 2, 16
    N = limit // (S * M)
    assert S * M * N == limit
    assert lib.emu_workspace_bytes(M, N, S) == lib.EMU_NOALLOC_SCRATCH_BYTES
    assert _noalloc(lib, M=M, N=N + 16, split_S=S) == -3
    assert "static scratch" in lib.emu_last_error()
    assert _noalloc(lib, M=0, N=N + 16, split_S=S) == 0       # empty output: nothing to do
