"""The N > 1 host path on CPU: gloo ranks run the product function
``scaled_mm_column_sharded`` -- column slabs, one per rank, computed independently
(here by the CPU oracle standing in for the CUDA GEMM, which needs a GPU) and
all-gathered -- and the gathered output equals the unsharded one bit for bit, with
an even (2 ranks) and an uneven (3 ranks) split of N; the timed region's maximum
over ranks is taken correctly."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_exact_fp8_gb300.sharding import column_slab, max_over_ranks, scaled_mm_column_sharded


def test_column_slabs_partition_N():
    for N in (0, 16, 48, 5760, 1920, 256):
        for world in (1, 2, 3, 4, 8):
            slabs = [column_slab(N, r, world) for r in range(world)]
            assert slabs[0][0] == 0 and slabs[-1][1] == N
            for (a0, a1), (b0, b1) in zip(slabs, slabs[1:]):
                assert a1 == b0
            for n0, n1 in slabs:
                assert n0 % 16 == 0 and n1 % 16 == 0 and n1 >= n0
            widths = [n1 - n0 for n0, n1 in slabs]
            assert max(widths) - min(widths) <= 16
    with pytest.raises(ValueError):
        column_slab(40, 0, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_gemm(cs):
    """A CPU stand-in for api.scaled_mm with its argument set: the oracle on the
    slab's codes, returned as a bf16 tensor of the oracle's bits."""
    import oracle

    def compute(mat1, mat2_slab, scale_a, scale_b, **kw):
        a = mat1.view(torch.uint8).numpy()
        b = mat2_slab.t().contiguous().view(torch.uint8).numpy()       # [n, K] bytes
        y = oracle.scaled_mm(a, b, cs.fmt_a, cs.fmt_b, float(scale_a), float(scale_b),
                             cs.out_dtype, kw["use_fast_accum"], kw["splitk"], kw["preset"],
                             nthreads=1)
        return torch.from_numpy(y.view(np.int16).copy()).view(torch.bfloat16)
    return compute


def _worker(rank, world, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from bit_exact_fp8_gb300 import workloads as W
        cs = W.shrink(W.case("splitk-hopper-S2-slow-bf16"), 8, 112, 1024)   # 7 slabs of 16
        a, b = W.make_inputs(cs)
        x = torch.from_numpy(a).view(torch.float8_e4m3fn)
        w = torch.from_numpy(b).view(torch.float8_e4m3fn)                   # [N, K]
        sa = torch.tensor(cs.scale_a)
        sb = torch.tensor(cs.scale_b)
        full = scaled_mm_column_sharded(x, w.t(), sa, sb, compute=_oracle_gemm(cs),
                                        out_dtype=torch.bfloat16, use_fast_accum=cs.fast_accum,
                                        splitk=cs.split_S, preset=cs.preset)
        local = scaled_mm_column_sharded(x, w.t(), sa, sb, compute=_oracle_gemm(cs),
                                         gather=False, out_dtype=torch.bfloat16,
                                         use_fast_accum=cs.fast_accum, splitk=cs.split_S,
                                         preset=cs.preset)
        n0, n1 = column_slab(cs.N, rank, world)
        t_max = max_over_ranks(1.0 + rank)
        want = oracle.scaled_mm(a, b, cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b,
                                cs.out_dtype, cs.fast_accum, cs.split_S, cs.preset, nthreads=1)
        got = full.view(torch.int16).numpy().view(np.uint16)
        ok = (np.array_equal(got, want) and local.shape == (cs.M, n1 - n0)
              and np.array_equal(local.view(torch.int16).numpy().view(np.uint16), want[:, n0:n1]))
        with open(f"{result_path}.{rank}", "w") as f:
            f.write(f"{int(ok)} {t_max} {n1 - n0}")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", (2, 3))
def test_gloo_ranks_shard_by_columns_bit_identically(tmp_path, world):
    result = tmp_path / "result"
    mp.start_processes(_worker, args=(world, _free_port(), str(result)), nprocs=world,
                       join=True, start_method="spawn")
    widths = []
    for r in range(world):
        ok, t_max, width = (tmp_path / f"result.{r}").read_text().split()
        assert ok == "1", f"rank {r}"
        assert float(t_max) == float(world)
        widths.append(int(width))
    assert sum(widths) == 112 and (world == 2 or len(set(widths)) == 2)
