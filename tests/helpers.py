"""Shared helpers of the test suite: run one workload case through the CUDA path
(C ABI via the package's binding) and through the CPU oracle, as bit patterns."""
from __future__ import annotations

import numpy as np
import torch

import oracle

TORCH_FP8 = {"e4m3fn": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
TORCH_OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16,
             "e4m3fn": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def out_bits(y: torch.Tensor) -> np.ndarray:
    y = y.cpu()
    if y.dtype == torch.float32:
        return y.view(torch.int32).numpy().view(np.uint32)
    if y.element_size() == 1:
        return y.view(torch.uint8).numpy().copy()
    return y.view(torch.int16).numpy().view(np.uint16)


def gpu_run(cs, a: np.ndarray, b: np.ndarray, *, out=None, splitk=None, preset=None,
            device="cuda:0", prefill=None):
    """Run the case on the GPU through the package API; returns output bits."""
    from bit_exact_fp8_gb300 import scaled_mm
    dev = torch.device(device)
    A = torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(TORCH_FP8[cs.fmt_a])
    Bt = torch.from_numpy(np.ascontiguousarray(b)).to(dev).view(TORCH_FP8[cs.fmt_b])
    sa = torch.tensor(cs.scale_a, dtype=torch.float32, device=dev)
    sb = torch.tensor(cs.scale_b, dtype=torch.float32, device=dev)
    od = TORCH_OUT[cs.out_dtype]
    if out is None and prefill is not None:
        out = torch.empty((a.shape[0], b.shape[0]), dtype=od, device=dev)
        out.view(torch.uint8).fill_(prefill)
    sr = None if cs.scale_result is None else torch.tensor(cs.scale_result, dtype=torch.float32,
                                                            device=dev)
    y = scaled_mm(A, Bt.t(), sa, sb, scale_result=sr, out_dtype=od, use_fast_accum=cs.fast_accum,
                  splitk=cs.split_S if splitk is None else splitk,
                  preset=cs.preset if preset is None else preset, out=out)
    torch.cuda.synchronize()
    return out_bits(y)


def oracle_full(cs, a, b, preset=None):
    return oracle.scaled_mm(a, b, cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b, cs.out_dtype,
                            cs.fast_accum, cs.split_S, cs.preset if preset is None else preset,
                            scale_result=cs.scale_result)


def oracle_sampled(cs, a, b, im, jn, preset=None):
    acc = oracle.acc_sampled(a, b, cs.fmt_a, cs.fmt_b, im, jn, cs.fast_accum, cs.split_S,
                             cs.preset if preset is None else preset)
    return oracle.epilogue(acc, cs.scale_a, cs.scale_b, cs.out_dtype, scale_result=cs.scale_result)


def sample_indices(M: int, N: int, count: int, seed: int = 0):
    """Sampled outputs: the four corners, the last row and column, and random ones."""
    rng = np.random.default_rng(seed)
    im = list(rng.integers(0, M, count))
    jn = list(rng.integers(0, N, count))
    for m, n in ((0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)):
        im.append(m)
        jn.append(n)
    return np.array(im, np.int64), np.array(jn, np.int64)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = ""):
    """Bit-for-bit comparison (+0 != -0, NaN payloads count); reports the first few."""
    assert got.shape == want.shape, (got.shape, want.shape)
    bad = np.flatnonzero(got.ravel() != want.ravel())
    if bad.size:
        first = ", ".join(f"[{i}] got {int(got.ravel()[i]):#x} want {int(want.ravel()[i]):#x}"
                          for i in bad[:10])
        raise AssertionError(f"{what}: {bad.size} of {want.size} outputs differ: {first}")
