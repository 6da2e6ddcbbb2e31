"""The device entry point inside a captured CUDA graph: a launch-bound caller (small
shapes, many calls) captures scaled_mm once -- the tensor maps and launch
arguments are baked into the graph's nodes -- and replays it on new operands
written into the same device buffers.  Every replay must give the bits of a
direct call on those operands."""
import numpy as np
import pytest
import torch

from bit_exact_fp8_gb300 import workloads as W
from helpers import TORCH_FP8, TORCH_OUT, gpu_run, out_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cs", [W.case("tiny"),
                                W.shrink(W.case("splitk-hopper-S8-fast-bf16"), 16, 128, 4096)],
                         ids=lambda c: c.name)
def test_captured_graph_replays_bit_exactly(cs):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_exact_fp8_gb300 import build, scaled_mm
    build.build()
    dev = torch.device("cuda:0")
    od = TORCH_OUT[cs.out_dtype]
    A = torch.empty((cs.M, cs.K), dtype=torch.uint8, device=dev)
    B = torch.empty((cs.N, cs.K), dtype=torch.uint8, device=dev)
    sa = torch.tensor(cs.scale_a, dtype=torch.float32, device=dev)
    sb = torch.tensor(cs.scale_b, dtype=torch.float32, device=dev)
    out = torch.empty((cs.M, cs.N), dtype=od, device=dev)

    def call():
        scaled_mm(A.view(TORCH_FP8[cs.fmt_a]), B.view(TORCH_FP8[cs.fmt_b]).t(), sa, sb,
                  out_dtype=od, use_fast_accum=cs.fast_accum, splitk=cs.split_S,
                  preset=cs.preset, out=out)

    a0, b0 = W.make_inputs(cs)
    A.copy_(torch.from_numpy(a0))
    B.copy_(torch.from_numpy(b0))
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):                  # warm-up outside the capture
        call()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for seed in (11, 12, 13):
        cs_i = W.Case(cs.name, cs.M, cs.N, cs.K, cs.fmt_a, cs.fmt_b, cs.out_dtype,
                      fast_accum=cs.fast_accum, split_S=cs.split_S, preset=cs.preset, seed=seed,
                      scale_a=cs.scale_a, scale_b=cs.scale_b)
        a, b = W.make_inputs(cs_i)
        A.copy_(torch.from_numpy(a))
        B.copy_(torch.from_numpy(b))
        out.view(torch.uint8).fill_(0xA5)
        graph.replay()
        torch.cuda.synchronize(dev)
        assert np.array_equal(out_bits(out), gpu_run(cs_i, a, b)), f"replay with seed {seed}"
