"""The tensor cores as a source of exact products: the self-test behind the opt-in
tensor-core W tile ("User guide" section 6: the tensor-core kernels rest on what the
tensor cores compute; the one property used here is that a bf16 x bf16 product of two
pre-scaled FP8 values, alone in its output, comes back exact in fp32), and that tile
inside a captured CUDA graph."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_tensor_core_products_are_exact():
    import __graft_entry__
    __graft_entry__.build()
    from bit_exact_fp8_gb300 import _lib
    assert _lib.emu_tc_selftest() == 0
    assert _lib.emu_device_status() == 0


# with EMU_FP8_TC=1 (read once per process): the first call decides the gate outside any
# capture, then a captured call replays on new operands; every replay must give the
# oracle's bits
GRAPH_CHILD = r'''
import sys
sys.path.insert(0, "tests")
import numpy as np, torch
from bit_exact_fp8_gb300 import workloads as W, scaled_mm, _lib
from helpers import TORCH_FP8, TORCH_OUT, out_bits, oracle_full, assert_bits_equal
dev = torch.device("cuda:0")
cs = W.Case("tc-graph", 200, 96, 320, "e4m3fn", "e4m3fn", "bf16", fast_accum=True, split_S=1, seed=21)
od = TORCH_OUT[cs.out_dtype]
A = torch.empty((cs.M, cs.K), dtype=torch.uint8, device=dev)
B = torch.empty((cs.N, cs.K), dtype=torch.uint8, device=dev)
sa = torch.tensor(cs.scale_a, dtype=torch.float32, device=dev)
sb = torch.tensor(cs.scale_b, dtype=torch.float32, device=dev)
out = torch.empty((cs.M, cs.N), dtype=od, device=dev)
def call():
    scaled_mm(A.view(TORCH_FP8[cs.fmt_a]), B.view(TORCH_FP8[cs.fmt_b]).t(), sa, sb,
              out_dtype=od, use_fast_accum=cs.fast_accum, splitk=1, preset=cs.preset, out=out)
a0, b0 = W.make_inputs(cs)
A.copy_(torch.from_numpy(a0)); B.copy_(torch.from_numpy(b0))
side = torch.cuda.Stream(dev)
side.wait_stream(torch.cuda.current_stream(dev))
with torch.cuda.stream(side):
    call()
torch.cuda.current_stream(dev).wait_stream(side)
torch.cuda.synchronize(dev)
assert_bits_equal(out_bits(out), oracle_full(cs, a0, b0), "direct call")
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph):
    call()
for seed in (31, 32):
    cs_i = W.Case(cs.name, cs.M, cs.N, cs.K, cs.fmt_a, cs.fmt_b, cs.out_dtype,
                  fast_accum=True, split_S=1, seed=seed)
    a, b = W.make_inputs(cs_i)
    A.copy_(torch.from_numpy(a)); B.copy_(torch.from_numpy(b))
    out.view(torch.uint8).fill_(0xA5)
    graph.replay()
    torch.cuda.synchronize(dev)
    assert_bits_equal(out_bits(out), oracle_full(cs_i, a, b), f"replay {seed}")
assert _lib.emu_device_status() == 0
print("ok")
'''


def test_tensor_core_tile_in_a_captured_graph():
    import __graft_entry__
    __graft_entry__.build()
    env = dict(os.environ, EMU_FP8_TILE="W", EMU_FP8_TC="1")
    r = subprocess.run([sys.executable, "-c", GRAPH_CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]
