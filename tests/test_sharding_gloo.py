"""The N > 1 host path on CPU: two gloo ranks shard the GEMM by column slabs,
compute their slabs independently (here with the CPU oracle, as the CUDA path
needs a GPU) and all-gather them; the gathered output equals the unsharded one
bit for bit, and the timed region's maximum over ranks is taken correctly."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_exact_fp8_gb300.sharding import column_slab, gather_columns, max_over_ranks


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


def _worker(rank, world, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from bit_exact_fp8_gb300 import workloads as W
        cs = W.shrink(W.case("linear"), 8, 96, 256)
        a, b = W.make_inputs(cs)
        n0, n1 = column_slab(cs.N, rank, world)
        local = oracle.scaled_mm(a, b[n0:n1], cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b,
                                 cs.out_dtype, cs.fast_accum, cs.split_S, cs.preset, nthreads=1)
        local_t = torch.from_numpy(local.view(np.int16).copy()).view(torch.bfloat16)
        full = gather_columns(local_t, cs.N)
        t_max = max_over_ranks(1.0 + rank)
        if rank == 0:
            want = oracle.scaled_mm(a, b, cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b,
                                    cs.out_dtype, cs.fast_accum, cs.split_S, cs.preset, nthreads=1)
            ok = np.array_equal(full.view(torch.int16).numpy().view(np.uint16), want)
            with open(result_path, "w") as f:
                f.write(f"{int(ok)} {t_max}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_gather_bit_identically(tmp_path):
    world = 2
    result = tmp_path / "result.txt"
    mp.start_processes(_worker, args=(world, _free_port(), str(result)), nprocs=world,
                       join=True, start_method="spawn")
    ok, t_max = result.read_text().split()
    assert ok == "1"
    assert float(t_max) == 2.0
