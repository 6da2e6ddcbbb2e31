"""torch-facing API: ``scaled_mm`` with the argument set of torch 2.7.1
``torch._scaled_mm`` ("User guide", section 3 "A first GEMM": same names, order and
defaults; mat2 is [K, N] column-major, e.g. ``w.t()``), plus the explicit split.

PyTorch provides device memory and the stream only; the GEMM runs in libemufp8's
CUDA kernels.  Tensors must be on a CUDA device: there is no CPU path.
"""
from __future__ import annotations

from typing import Optional, Union

import torch

from . import _lib

_FMT = {torch.float8_e4m3fn: _lib.EMU_E4M3FN, torch.float8_e5m2: _lib.EMU_E5M2}
_OUT = {torch.float32: _lib.EMU_OUT_F32, torch.bfloat16: _lib.EMU_OUT_BF16,
        torch.float16: _lib.EMU_OUT_F16, torch.float8_e4m3fn: _lib.EMU_OUT_E4M3FN,
        torch.float8_e5m2: _lib.EMU_OUT_E5M2}


class EmuError(Exception):
    """Base class of this package's errors."""


class ReferenceRejectsError(EmuError, RuntimeError):
    """torch 2.7.1 or the reference cuBLAS would reject the call (layout,
    divisibility, dtypes) -- "User guide", section 9 "Errors and warnings"."""


class UnsupportedFeatureError(EmuError, NotImplementedError):
    """bias, row-wise scales, grad mode, or a preset the kernels do not
    implement ("Limitations of mmaemu v0.1", table "Features outside v0.1")."""


class EmuCudaError(EmuError, RuntimeError):
    """a CUDA launch failed."""


def _raise(status: int, what: str):
    msg = f"{what}: {_lib.emu_last_error()}"
    if status == _lib.EMU_EREJECT:
        raise ReferenceRejectsError(msg)
    if status == _lib.EMU_EUNSUPPORTED:
        raise UnsupportedFeatureError(msg)
    if status == _lib.EMU_ECUDA:
        raise EmuCudaError(msg)
    raise ValueError(msg)


def preset_params(preset: Union[str, dict, "_lib.emu_preset_t"]) -> "_lib.emu_preset_t":
    if isinstance(preset, _lib.emu_preset_t):
        return preset
    if isinstance(preset, str):
        return _lib.emu_preset_get(preset)
    return _lib.emu_preset_t(**preset)


def workspace_bytes(M: int, N: int, split_S: int) -> int:
    return _lib.emu_workspace_bytes(M, N, split_S)


def tile_for(M: int, N: int, K: int, *, use_fast_accum: bool = False, splitk: int = 1,
             preset: Union[str, dict, "_lib.emu_preset_t"] = "hopper", sm_count: int = 0) -> str:
    """Name of the CTA tile ``scaled_mm`` launches for an (M, N, K) problem ("none"
    when nothing is launched); ``sm_count`` > 0 stands in for the device's."""
    st, name = _lib.emu_tile_for(M, N, K, int(use_fast_accum), splitk, preset_params(preset),
                                 sm_count)
    if st != _lib.EMU_OK:
        _raise(st, "tile_for")
    return name


def scaled_mm(mat1: torch.Tensor, mat2: torch.Tensor, scale_a: torch.Tensor,
              scale_b: torch.Tensor, bias: Optional[torch.Tensor] = None,
              scale_result: Optional[torch.Tensor] = None,
              out_dtype: Optional[torch.dtype] = None, use_fast_accum: bool = False, *,
              splitk: int = 1, preset="hopper", out: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Emulated ``torch._scaled_mm(mat1, mat2, scale_a, scale_b, ...)``.

    mat1 [M,K] row-major and mat2 [K,N] column-major FP8 tensors on one CUDA
    device, scale_a/scale_b one-element fp32 tensors there.  ``splitk`` is the
    explicit split-K factor S, ``preset`` "hopper" (default) or "ada" or a
    parameter dict.  Returns out [M,N] (out_dtype defaults to mat1's dtype, as in
    torch; an FP8 out_dtype takes the optional one-element ``scale_result``)."""
    if bias is not None:
        raise UnsupportedFeatureError("bias is not supported (it raises on the reference too)")
    if torch.is_grad_enabled() and any(t.requires_grad for t in (mat1, mat2)):
        raise UnsupportedFeatureError("inference only: inputs require grad under grad mode")
    if mat1.dim() != 2 or mat2.dim() != 2:
        raise ValueError("mat1 and mat2 must be 2-D")
    if mat1.dtype not in _FMT or mat2.dtype not in _FMT:
        raise ReferenceRejectsError(f"FP8 operands expected, got {mat1.dtype}, {mat2.dtype}")
    if not (mat1.is_cuda and mat2.is_cuda and scale_a.is_cuda and scale_b.is_cuda):
        raise ValueError("all tensors must be on a CUDA device (there is no CPU path)")
    dev = mat1.device
    if mat2.device != dev or scale_a.device != dev or scale_b.device != dev:
        raise ValueError("all tensors must be on the same device")
    M, K = mat1.shape
    K2, N = mat2.shape
    if K != K2:
        raise ValueError(f"shape mismatch: {tuple(mat1.shape)} @ {tuple(mat2.shape)}")
    if mat1.numel() > 0 and not mat1.is_contiguous():
        raise ReferenceRejectsError("mat1 must be row-major")
    if mat2.numel() > 0 and not (mat2.stride(0) == 1 and (mat2.stride(1) == K or N <= 1)):
        raise ReferenceRejectsError("mat2 must be column-major ([K, N] with K contiguous, e.g. w.t())")
    if scale_result is not None and (not scale_result.is_cuda or scale_result.device != dev
                                     or scale_result.numel() != 1
                                     or scale_result.dtype != torch.float32):
        raise ValueError("scale_result must be a one-element float32 tensor on the device")
    for name, sc in (("scale_a", scale_a), ("scale_b", scale_b)):
        if sc.numel() != 1:
            raise UnsupportedFeatureError(f"row-wise {name} is not supported (tensor-wise only)")
        if sc.dtype != torch.float32:
            raise ReferenceRejectsError(f"{name} must be float32")
    if out_dtype is None:
        out_dtype = mat1.dtype
    if out_dtype not in _OUT:
        raise UnsupportedFeatureError(f"out_dtype {out_dtype} is not supported")
    P = preset_params(preset)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    elif out.shape != (M, N) or out.dtype != out_dtype or not out.is_contiguous() or out.device != dev:
        raise ValueError("out must be a contiguous [M, N] tensor of out_dtype on the device")
    need = _lib.emu_workspace_bytes(M, N, int(splitk))
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if (workspace is not None and need > 0) else 0
    ws_bytes = workspace.numel() * workspace.element_size() if (workspace is not None and need > 0) else 0
    stream = torch.cuda.current_stream(dev).cuda_stream
    sr_ptr = scale_result.data_ptr() if scale_result is not None else 0
    st = _lib.emu_scaled_mm_ex(mat1.data_ptr(), _FMT[mat1.dtype], mat2.data_ptr(),
                               _FMT[mat2.dtype], M, N, K, scale_a.data_ptr(), scale_b.data_ptr(),
                               sr_ptr, out.data_ptr(), _OUT[out_dtype], int(bool(use_fast_accum)),
                               int(splitk), P, ws_ptr, ws_bytes, stream)
    if st != _lib.EMU_OK:
        _raise(st, "emu_scaled_mm")
    return out


def staging_bytes(M: int, N: int, K: int, split_S: int, out_dtype: torch.dtype) -> int:
    """Device staging bytes scaled_mm_host needs for these sizes."""
    return _lib.emu_host_staging_bytes(M, N, K, split_S, _OUT[out_dtype])


def scaled_mm_host(mat1: torch.Tensor, mat2: torch.Tensor, scale_a: float, scale_b: float,
                   scale_result: Optional[float] = None, out_dtype: Optional[torch.dtype] = None,
                   use_fast_accum: bool = False, *, splitk: int = 1, preset="hopper",
                   out: Optional[torch.Tensor] = None, staging: Optional[torch.Tensor] = None,
                   chunks: int = 0, device=None, synchronize: bool = True) -> torch.Tensor:
    """``scaled_mm`` on HOST tensors: mat1 [M,K] row-major and mat2 [K,N]
    column-major FP8 tensors in host memory (pinned, e.g. ``.pin_memory()``, for
    the copies to overlap the compute), scales as Python floats.  The library
    uploads the operands in ``chunks`` column slabs (0: one per 64 MiB of B),
    computes each slab as soon as it has landed and copies the result back, on its own streams ordered after the
    current stream of ``device``; the bits equal those of ``scaled_mm``.  Returns
    the host [M,N] result (``out`` if given, pinned); with ``synchronize=False`` it
    is valid only once the device's current stream has completed."""
    if mat1.dim() != 2 or mat2.dim() != 2:
        raise ValueError("mat1 and mat2 must be 2-D")
    if mat1.dtype not in _FMT or mat2.dtype not in _FMT:
        raise ReferenceRejectsError(f"FP8 operands expected, got {mat1.dtype}, {mat2.dtype}")
    if mat1.is_cuda or mat2.is_cuda:
        raise ValueError("scaled_mm_host takes host tensors (use scaled_mm for device tensors)")
    M, K = mat1.shape
    K2, N = mat2.shape
    if K != K2:
        raise ValueError(f"shape mismatch: {tuple(mat1.shape)} @ {tuple(mat2.shape)}")
    if mat1.numel() > 0 and not mat1.is_contiguous():
        raise ReferenceRejectsError("mat1 must be row-major")
    if mat2.numel() > 0 and not (mat2.stride(0) == 1 and (mat2.stride(1) == K or N <= 1)):
        raise ReferenceRejectsError("mat2 must be column-major ([K, N] with K contiguous, e.g. w.t())")
    if out_dtype is None:
        out_dtype = mat1.dtype
    if out_dtype not in _OUT:
        raise UnsupportedFeatureError(f"out_dtype {out_dtype} is not supported")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    P = preset_params(preset)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, pin_memory=True)
    elif out.shape != (M, N) or out.dtype != out_dtype or not out.is_contiguous() or out.is_cuda:
        raise ValueError("out must be a contiguous host [M, N] tensor of out_dtype")
    need = _lib.emu_host_staging_bytes(M, N, K, int(splitk), _OUT[out_dtype])
    if staging is None or staging.numel() * staging.element_size() < need or staging.data_ptr() % 256:
        staging = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        st = _lib.emu_scaled_mm_host(mat1.data_ptr(), _FMT[mat1.dtype], mat2.data_ptr(),
                                     _FMT[mat2.dtype], M, N, K, scale_a, scale_b, scale_result,
                                     out.data_ptr(), _OUT[out_dtype], int(bool(use_fast_accum)),
                                     int(splitk), P, staging.data_ptr(),
                                     staging.numel() * staging.element_size(), int(chunks),
                                     stream.cuda_stream)
        if st != _lib.EMU_OK:
            _raise(st, "emu_scaled_mm_host")
        if synchronize:
            stream.synchronize()
    return out


def accumulate(x: torch.Tensor, w: torch.Tensor, use_fast_accum: bool, *, splitk: int = 1,
               preset="hopper") -> torch.Tensor:
    """The fp32 accumulator before the scales ("User guide", section 3: both operands
    as [rows, K]; no default for use_fast_accum).  Equal to the fp32 output with unit
    scales, since the accumulator is never -0."""
    one = torch.ones((), dtype=torch.float32, device=x.device)
    return scaled_mm(x, w.t(), one, one, out_dtype=torch.float32, use_fast_accum=use_fast_accum,
                     splitk=splitk, preset=preset)
