"""emu_scaled_mm_host: the GEMM with host operands and result, uploads, slab GEMMs
and copies back overlapped on the library's streams.  Every output depends only on
its row of A and column of B, so for any slab count the bits must equal those of
the device entry point (and of the oracle where it runs the whole case): bit-exact,
the tolerance of every parity test here."""
import dataclasses

import numpy as np
import pytest
import torch

from bit_exact_fp8_gb300 import workloads as W
from helpers import TORCH_FP8, TORCH_OUT, assert_bits_equal, gpu_run, oracle_full, out_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_exact_fp8_gb300 import build
    build.build()


def host_run(cs, a, b, chunks, staging=None):
    from bit_exact_fp8_gb300 import scaled_mm_host
    A = torch.from_numpy(np.ascontiguousarray(a)).view(TORCH_FP8[cs.fmt_a]).pin_memory()
    Bt = torch.from_numpy(np.ascontiguousarray(b)).view(TORCH_FP8[cs.fmt_b]).pin_memory()
    od = TORCH_OUT[cs.out_dtype]
    out = torch.empty((a.shape[0], b.shape[0]), dtype=od).pin_memory()
    out.view(torch.uint8).fill_(0xA5)                       # stale bytes must be overwritten
    y = scaled_mm_host(A, Bt.t(), cs.scale_a, cs.scale_b, scale_result=cs.scale_result,
                       out_dtype=od, use_fast_accum=cs.fast_accum, splitk=cs.split_S,
                       preset=cs.preset, out=out, staging=staging, chunks=chunks,
                       device="cuda:0")
    return out_bits(y)


SMALL = [
    W.case("tiny"),
    W.shrink(W.case("linear"), 48, 1440, 512),
    dataclasses.replace(W.shrink(W.case("linear"), 40, 496, 320), fast_accum=False, preset="ada"),
    W.shrink(W.case("splitk-hopper-S8-fast-bf16"), 16, 256, 8192),
    W.shrink(W.case("splitk-ada-S8-slow-f32"), 16, 128, 4096 + 64),
    dataclasses.replace(W.shrink(W.case("linear"), 32, 160, 256), out_dtype="e4m3fn",
                        scale_result=0.37),
]


@pytest.mark.parametrize("cs", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("chunks", [1, 3, 4, 0, 16])
def test_host_path_matches_oracle_and_device_path(cs, chunks):
    a, b = W.make_inputs(cs)
    got = host_run(cs, a, b, chunks)
    assert_bits_equal(got, gpu_run(cs, a, b), f"{cs.name} host vs device, chunks={chunks}")
    if chunks == 3:
        assert_bits_equal(got, oracle_full(cs, a, b), f"{cs.name} host vs oracle")


def test_host_path_full_linear_and_reused_staging():
    from bit_exact_fp8_gb300 import staging_bytes
    cs = W.case("linear")
    a, b = W.make_inputs(cs)
    want = gpu_run(cs, a, b)
    need = staging_bytes(cs.M, cs.N, cs.K, cs.split_S, TORCH_OUT[cs.out_dtype])
    staging = torch.empty(need, dtype=torch.uint8, device="cuda:0")
    for chunks in (4, 6):
        staging.fill_(0x5A)
        assert_bits_equal(host_run(cs, a, b, chunks, staging=staging), want,
                          f"linear host, chunks={chunks}")


def test_host_path_k0_and_empty():
    from bit_exact_fp8_gb300 import scaled_mm_host
    x = torch.empty((16, 0), dtype=torch.float8_e4m3fn).pin_memory()
    w = torch.empty((64, 0), dtype=torch.float8_e4m3fn).pin_memory()
    y = scaled_mm_host(x, w.t(), 2.0, 3.0, out_dtype=torch.float32)
    assert y.shape == (16, 64)
    assert (y.view(torch.int32) == 0).all()                 # fma(+0, alpha, +0) = +0
    e = scaled_mm_host(torch.empty((0, 32), dtype=torch.float8_e4m3fn),
                       torch.empty((16, 32), dtype=torch.float8_e4m3fn).t(), 1.0, 1.0,
                       out_dtype=torch.bfloat16)
    assert e.shape == (0, 16)
