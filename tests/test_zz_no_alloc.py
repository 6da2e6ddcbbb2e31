"""emu_scaled_mm_noalloc: the entry point for callers that cannot allocate device
memory (a plugin interface that hands over only inputs and outputs, memory fixed at
start-up, a host framework that owns every allocation).  It keeps the split-K
partials in the library's static device scratch instead of a caller workspace.

Called through the C ABI binding, it must return the same bits as emu_scaled_mm
with a caller-allocated workspace, and as the CPU oracle (bit-exact, the tolerance
of every parity test here), on two calls in a row, since each call reuses the
scratch the previous call left behind.  One case fills the scratch exactly
(split_S * M * N == EMU_NOALLOC_SCRATCH_BYTES / 4).  This file is collected last,
and passes alone in a fresh process as well as after the other tests."""
import numpy as np
import pytest
import torch

from bit_exact_fp8_gb300 import workloads as W

pytestmark = pytest.mark.gpu

FMT = {"e4m3fn": 0, "e5m2": 1}
OUT = {"f32": (0, torch.float32), "bf16": (1, torch.bfloat16), "f16": (2, torch.float16)}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_exact_fp8_gb300 import _lib, build
    build.build()
    return _lib


def _bits(t):
    t = t.cpu()
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16).numpy().copy()


CASES = [
    W.shrink(W.case("splitk-hopper-S24-fast-f32"), 16, 256, 16384),
    W.shrink(W.case("splitk-ada-S8-slow-bf16"), 16, 256, 16384 + 64),
    W.shrink(W.case("splitk-hopper-S2-slow-f32"), 48, 112, 4096 + 16),
    W.case("splitk-ada-S24-fast-f32"),                       # full size, 393 KB of partials
    W.case("tiny"),                                          # S = 1: no scratch at all
    # the partials fill the 4 MiB scratch exactly: 2 x 16 x 32768 fp32
    W.shrink(W.case("splitk-hopper-S2-fast-bf16"), 16, 32768, 2048),
]


@pytest.mark.parametrize("cs", CASES, ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point_twice(lib, cs):
    dev = torch.device("cuda:0")
    a, b = W.make_inputs(cs)
    A = torch.from_numpy(a).to(dev)
    B = torch.from_numpy(b).to(dev)
    sa = torch.tensor(cs.scale_a, dtype=torch.float32, device=dev)
    sb = torch.tensor(cs.scale_b, dtype=torch.float32, device=dev)
    odc, odt = OUT[cs.out_dtype]
    preset = lib.emu_preset_get(cs.preset)
    stream = torch.cuda.current_stream(dev).cuda_stream
    need = lib.emu_workspace_bytes(cs.M, cs.N, cs.split_S)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

    ref = torch.empty((cs.M, cs.N), dtype=odt, device=dev)
    st = lib.emu_scaled_mm(A.data_ptr(), FMT[cs.fmt_a], B.data_ptr(), FMT[cs.fmt_b], cs.M, cs.N,
                           cs.K, sa.data_ptr(), sb.data_ptr(), ref.data_ptr(), odc,
                           int(cs.fast_accum), cs.split_S, preset, ws.data_ptr(), ws.numel(),
                           stream)
    assert st == 0, lib.emu_last_error()
    want = _bits(ref)
    import oracle
    orc = oracle.scaled_mm(a, b, cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b, cs.out_dtype,
                           cs.fast_accum, cs.split_S, cs.preset)
    orc = orc.view(np.int32 if cs.out_dtype == "f32" else np.int16)
    bad = np.flatnonzero(orc.ravel() != want.ravel())
    assert bad.size == 0, f"emu_scaled_mm vs oracle: {bad.size} outputs differ, first at {bad[:5]}"

    for call in range(2):
        out = torch.empty((cs.M, cs.N), dtype=odt, device=dev)
        out.view(torch.uint8).fill_(0xFF if call == 0 else 0x5A)
        st = lib.emu_scaled_mm_noalloc(A.data_ptr(), FMT[cs.fmt_a], B.data_ptr(), FMT[cs.fmt_b],
                                       cs.M, cs.N, cs.K, sa.data_ptr(), sb.data_ptr(),
                                       out.data_ptr(), odc, int(cs.fast_accum), cs.split_S,
                                       preset, stream)
        assert st == 0, lib.emu_last_error()
        torch.cuda.synchronize(dev)
        got = _bits(out)
        bad = np.flatnonzero(got.ravel() != want.ravel())
        assert bad.size == 0, f"call {call}: {bad.size} outputs differ, first at {bad[:5]}"


def test_noalloc_rejects_partials_beyond_the_static_scratch(lib):
    # split_S * M * N above EMU_NOALLOC_SCRATCH_BYTES / 4: refused before any launch
    preset = lib.emu_preset_get("hopper")
    fake = 1 << 20
    M, N, S = 1024, 1024, 2
    assert S * M * N * 4 > lib.EMU_NOALLOC_SCRATCH_BYTES
    st = lib.emu_scaled_mm_noalloc(fake, 0, fake, 0, M, N, 4096, fake, fake, fake, 0, 1, S,
                                   preset, 0)
    assert st == -3
    assert "static scratch" in lib.emu_last_error()
