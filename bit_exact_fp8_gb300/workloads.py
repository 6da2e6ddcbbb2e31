"""Seeded synthetic inputs for the emulated FP8 GEMM workloads.

This module only draws random FP8 codes; it holds none of the GEMM's arithmetic,
so both the CUDA path and the CPU oracle take their inputs from it.

The value distributions follow the documentation's own example ("User guide",
section 3 "A first GEMM": x = (randn(64, 1920) * 40).clamp(-448, 448) cast to
E4M3, then w = (randn(5760, 1920) * 40).clamp(...) from the same seed-0 stream;
tensor-wise scales 1/64 and 1/32).  No public dataset is named by the pages; the
Evo 2 projections the pages benchmark (an M x 5760 x 1920 linear layer) are
stood in for by the linear-layer and projection-batch shapes below.

Every array is returned as raw FP8 codes (numpy uint8):
  a  [M, K]  mat1, row-major
  b  [N, K]  the bytes of mat2 [K, N] column-major (w.t() of a row-major [N, K])
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, List, Optional

import numpy as np
import torch

FP8_MAX = {"e4m3fn": 448.0, "e5m2": 57344.0}
# largest finite code magnitudes: E4M3FN 0.1111.110, E5M2 0.11110.11
FP8_MAX_CODE = {"e4m3fn": 0x7E, "e5m2": 0x7B}
FP8_FRAC_BITS = {"e4m3fn": 3, "e5m2": 2}
_TORCH_FP8 = {"e4m3fn": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _cast_codes(x: torch.Tensor, fmt: str) -> np.ndarray:
    """fp32 tensor -> FP8 codes through torch's own cast (round to nearest even)."""
    return x.to(_TORCH_FP8[fmt]).view(torch.uint8).numpy().copy()


def gaussian_codes(gen: torch.Generator, rows: int, cols: int, scale: float, fmt: str) -> np.ndarray:
    x = (torch.randn(rows, cols, generator=gen) * scale).clamp(-FP8_MAX[fmt], FP8_MAX[fmt])
    return _cast_codes(x, fmt)


def mixed_codes(gen: torch.Generator, rows: int, cols: int, fmt: str, alternate_max_sign: bool) -> np.ndarray:
    """Adversarial mix along K: 70% (randn*40) clamped and cast, 10% subnormal codes
    (uniform over the format's subnormal fractions, random sign), 10% exact zeros
    (+0 or -0 codes), 10% +-max; with alternate_max_sign the max entries take the
    sign (-1)^k, so that max x max products cancel inside a block."""
    base = gaussian_codes(gen, rows, cols, 40.0, fmt)
    u = torch.rand(rows, cols, generator=gen).numpy()
    fb = FP8_FRAC_BITS[fmt]
    sub_frac = torch.randint(1, 1 << fb, (rows, cols), generator=gen).numpy().astype(np.uint8)
    sign = (torch.randint(0, 2, (rows, cols), generator=gen).numpy().astype(np.uint8) << 7)
    out = base.copy()
    sub = (u >= 0.70) & (u < 0.80)
    zer = (u >= 0.80) & (u < 0.90)
    mx = u >= 0.90
    out[sub] = (sign | sub_frac)[sub]
    out[zer] = sign[zer]
    if alternate_max_sign:
        kpar = (np.arange(cols) & 1).astype(np.uint8) << 7
        mx_codes = np.broadcast_to(kpar, (rows, cols)) | FP8_MAX_CODE[fmt]
    else:
        mx_codes = np.full((rows, cols), FP8_MAX_CODE[fmt], dtype=np.uint8)
    out[mx] = mx_codes[mx]
    return out


@dataclass(frozen=True)
class Case:
    """One GEMM call of a workload: shapes, formats, epilogue, accumulation, split."""
    name: str
    M: int
    N: int
    K: int
    fmt_a: str = "e4m3fn"
    fmt_b: str = "e4m3fn"
    out_dtype: str = "bf16"
    fast_accum: bool = True
    split_S: int = 1
    preset: str = "hopper"
    scale_a: float = 1.0 / 64
    scale_b: float = 1.0 / 32
    gen: str = "gauss"          # "gauss" | "mixed"
    seed: int = 0
    sigma_a: float = 40.0
    sigma_b: float = 40.0
    scale_result: Optional[float] = None   # fp8 outputs: multiplier after the scales

    @property
    def macs(self) -> int:
        return self.M * self.N * self.K


def make_inputs(case: Case, M: int | None = None, N: int | None = None, K: int | None = None):
    """Draw the case's operands (optionally at other sizes, same recipe).
    Returns (a [M,K] uint8, b [N,K] uint8)."""
    M = case.M if M is None else M
    N = case.N if N is None else N
    K = case.K if K is None else K
    gen = torch.Generator().manual_seed(case.seed)
    if case.gen == "gauss":
        a = gaussian_codes(gen, M, K, case.sigma_a, case.fmt_a)
        b = gaussian_codes(gen, N, K, case.sigma_b, case.fmt_b)
    elif case.gen == "mixed":
        a = mixed_codes(gen, M, K, case.fmt_a, alternate_max_sign=True)
        b = mixed_codes(gen, N, K, case.fmt_b, alternate_max_sign=False)
    else:
        raise ValueError(case.gen)
    return a, b


def _config_cases() -> Dict[str, List[Case]]:
    c: Dict[str, List[Case]] = {}
    # 1. tiny: M=16, N=64, K=256, seed 0, bf16, fast, S=1, hopper
    c["tiny"] = [Case("tiny", 16, 64, 256)]
    # 2. linear-layer shape of the user guide's example: M=64, K=1920, N=5760
    c["linear"] = [Case("linear", 64, 5760, 1920)]
    # 3. square 4096^3, adversarial mix, slow accumulation, three format pairs,
    #    fp32 and bf16 outputs (e5m2 x e5m2 is a rejection case, not a workload)
    sq = []
    for fa, fb in (("e4m3fn", "e4m3fn"), ("e4m3fn", "e5m2"), ("e5m2", "e4m3fn")):
        for od in ("f32", "bf16"):
            sq.append(Case(f"square-{fa}x{fb}-{od}", 4096, 4096, 4096, fa, fb, od,
                           fast_accum=False, gen="mixed", seed=3))
    c["square"] = sq
    # 4. split-K: M=16, N=256, K=262144, (randn*8) operands, S in {2, 8, 24}
    sk = []
    for preset in ("hopper", "ada"):
        for S in (2, 8, 24):
            for fast in (True, False):
                for od in ("bf16", "f32"):
                    sk.append(Case(f"splitk-{preset}-S{S}-{'fast' if fast else 'slow'}-{od}",
                                   16, 256, 262144, out_dtype=od, fast_accum=fast, split_S=S,
                                   preset=preset, seed=4, sigma_a=8.0, sigma_b=8.0))
    c["splitk"] = sk
    # 5. projection batch: M=8192 tokens, K=1920, N in {1920, 5760}
    c["projection"] = [Case(f"projection-N{N}", 8192, N, 1920, scale_a=1.0 / 128,
                            scale_b=1.0 / 64, seed=5, sigma_a=40.0, sigma_b=20.0)
                       for N in (1920, 5760)]
    return c


CONFIGS: Dict[str, List[Case]] = _config_cases()


def case(name: str) -> Case:
    for cases in CONFIGS.values():
        for cs in cases:
            if cs.name == name:
                return cs
    raise KeyError(name)


def shrink(cs: Case, M: int, N: int, K: int) -> Case:
    """The same recipe at smaller sizes (for oracle-sized parity runs)."""
    return replace(cs, name=f"{cs.name}@{M}x{N}x{K}", M=M, N=N, K=K)


def named(name: str) -> Case:
    """A workload case by name; "NAME@MxNxK" is case NAME's recipe at those sizes."""
    if "@" not in name:
        return case(name)
    base, sizes = name.split("@", 1)
    M, N, K = (int(v) for v in sizes.split("x"))
    return shrink(case(base), M, N, K)
