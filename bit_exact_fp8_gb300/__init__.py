"""bit_exact_fp8_gb300 -- the FP8 scaled GEMM of a reference tensor-core platform
(the mmaemu "hopper" and "ada" presets), computed bit for bit by hand-written
sm_103a CUDA kernels on a GB300.

    from bit_exact_fp8_gb300 import scaled_mm
    y = scaled_mm(x, w.t(), scale_x, scale_w, out_dtype=torch.bfloat16, use_fast_accum=True)

The C ABI is include/emu_fp8.h (libemufp8.so, built by ``build.build()``);
``_lib`` binds it through ctypes, ``api`` adds the torch-facing call.
"""
from .api import (EmuCudaError, EmuError, ReferenceRejectsError, UnsupportedFeatureError,
                  accumulate, preset_params, scaled_mm, scaled_mm_host, staging_bytes,
                  tile_for, workspace_bytes)

__all__ = ["scaled_mm", "scaled_mm_host", "accumulate", "preset_params", "workspace_bytes",
           "staging_bytes", "tile_for", "EmuError", "ReferenceRejectsError", "UnsupportedFeatureError",
           "EmuCudaError"]
