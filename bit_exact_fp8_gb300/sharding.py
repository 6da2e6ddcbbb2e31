"""Multi-GPU use of the emulated FP8 GEMM: one process per GPU (torch.distributed).

Every output (m, n) depends only on row m of A and column n of B, and a split-K
partition is fixed by S, not by the hardware.  So the GEMM shards by columns with
no exchange in the data path: each rank computes out[:, n0:n1] on its own GPU
from the full A and its slab of B, and the result is bit-identical to the
unsharded call by construction.  The only collective is the optional all-gather
of the output slabs, for callers that need the whole output on every rank.
"""
from __future__ import annotations

from typing import Callable, Optional, Tuple

import torch


def column_slab(N: int, rank: int, world: int, align: int = 16) -> Tuple[int, int]:
    """[n0, n1) of rank's slab: contiguous, in rank order, covering [0, N) exactly.

    Slab boundaries fall on multiples of ``align`` (16: the N % 16 rule of the
    reference's cuBLAS applies to every slab), and slab widths differ by at most
    ``align``.  Trailing ranks get an empty slab when N / align < world."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError(f"bad rank {rank} of {world}")
    if N < 0 or N % align:
        raise ValueError(f"N = {N} must be a non-negative multiple of {align}")
    units = N // align
    q, r = divmod(units, world)
    u0 = rank * q + min(rank, r)
    u1 = u0 + q + (1 if rank < r else 0)
    return u0 * align, u1 * align


def max_over_ranks(value: float, group=None) -> float:
    """The maximum of a host float over all ranks (e.g. the timed region)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return float(value)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def gather_columns(local: torch.Tensor, N: int, group=None) -> torch.Tensor:
    """All-gather the [M, n1 - n0] slabs of every rank into the full [M, N] output."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    M = local.shape[0]
    widths = [column_slab(N, r, world)[1] - column_slab(N, r, world)[0] for r in range(world)]
    wmax = max(widths) if widths else 0
    padded = torch.zeros((M, wmax), dtype=local.dtype, device=local.device)
    padded[:, :local.shape[1]] = local
    # gather raw bytes so every dtype (bf16, fp16, fp32) travels bit for bit
    flat = padded.contiguous().view(torch.uint8)
    parts = [torch.empty_like(flat) for _ in range(world)]
    dist.all_gather(parts, flat, group=group)
    out = torch.empty((M, N), dtype=local.dtype, device=local.device)
    for r in range(world):
        n0, n1 = column_slab(N, r, world)
        out[:, n0:n1] = parts[r].view(local.dtype).view(M, wmax)[:, :n1 - n0]
    return out


def scaled_mm_column_sharded(mat1: torch.Tensor, mat2: torch.Tensor, scale_a: torch.Tensor,
                             scale_b: torch.Tensor, *, group=None, gather: bool = True,
                             compute: Optional[Callable[..., torch.Tensor]] = None,
                             **kwargs) -> torch.Tensor:
    """This rank's share of ``scaled_mm(mat1, mat2, ...)``: its column slab of the
    output, computed on its own GPU; with ``gather`` the full output on every rank.

    ``compute`` is the per-rank GEMM, called as ``compute(mat1, mat2_slab, scale_a,
    scale_b, **kwargs)`` with the [K, n1 - n0] column-major slab of mat2; it defaults
    to ``api.scaled_mm`` (the CUDA path).  Another GEMM of the same argument set can
    stand in for it, e.g. on hosts without a GPU."""
    import torch.distributed as dist
    if compute is None:
        from .api import scaled_mm as compute
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    N = mat2.shape[1]
    n0, n1 = column_slab(N, rank, world)
    local = compute(mat1, mat2[:, n0:n1], scale_a, scale_b, **kwargs)
    if not gather or world == 1:
        return local
    return gather_columns(local, N, group)
