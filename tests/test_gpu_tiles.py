"""Every CTA tile shape of the GEMM kernel, forced one at a time through
EMU_FP8_TILE (read once per process, hence one subprocess per tile), is bit-exact
against the oracle on ragged shapes, both presets, fast and slow accumulation,
split-K, the three output dtypes, and Inf and NaN codes."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# "W:TC" is the W tile with its products from the tensor cores (opt-in, EMU_FP8_TC=1)
TILES = ["M40", "M32", "M64", "S", "K8", "K4", "K8H", "K4H", "C2", "C4", "C1", "C1L", "W", "W:TC"]

CHILD = r'''
import sys
sys.path.insert(0, "tests")
from bit_exact_fp8_gb300 import workloads as W
from helpers import assert_bits_equal, gpu_run, oracle_full
cases = [
    W.Case("t1", 70, 96, 528, "e4m3fn", "e4m3fn", "bf16", fast_accum=True, gen="mixed", seed=1),
    W.Case("t2", 33, 48, 1040, "e4m3fn", "e5m2", "f32", fast_accum=False, gen="mixed", seed=2),
    W.Case("t3", 16, 80, 4096 + 48, "e5m2", "e4m3fn", "f16", fast_accum=True, split_S=3, seed=3),
    W.Case("t4", 20, 64, 64 * 37 + 32, out_dtype="f32", fast_accum=False, split_S=5, preset="ada",
           seed=4, sigma_a=8.0, sigma_b=8.0),
    W.Case("t5", 130, 112, 256, out_dtype="bf16", fast_accum=False, preset="ada", gen="mixed", seed=5),
]
for cs in cases:
    a, b = W.make_inputs(cs)
    assert_bits_equal(gpu_run(cs, a, b), oracle_full(cs, a, b), cs.name)
# Inf and NaN codes: IEEE sums through every tile's block reduction
for fast, S in ((True, 1), (False, 2)):
    cs = W.Case("t6", 24, 32, 512, "e5m2", "e4m3fn", "f32", fast_accum=fast, split_S=S, seed=6)
    a, b = W.make_inputs(cs)
    a[2, 10] = 0x7C            # +Inf
    a[5, 11] = 0xFC            # -Inf
    a[5, 300] = 0x7C           # +Inf and -Inf in one row: NaN
    b[:, 60] = 0x00
    a[9, 60] = 0x7C            # Inf x 0: NaN
    a[13, 200] = 0x7E          # NaN code
    assert_bits_equal(gpu_run(cs, a, b), oracle_full(cs, a, b), f"t6 fast={fast} S={S}")
# an E4M3FN A with NaN codes against an E5M2 B with Inf and NaN codes (the W tile's
# tensor-core products: a NaN in A meets the expanded B's zeros)
for fast, S in ((True, 1), (True, 2)):
    cs = W.Case("t7", 140, 80, 576, "e4m3fn", "e5m2", "bf16", fast_accum=fast, split_S=S, seed=7)
    a, b = W.make_inputs(cs)
    a[3, 17] = 0x7F            # NaN
    a[100, 300] = 0xFF         # NaN
    b[5, 40] = 0x7C            # +Inf
    b[9, 41] = 0xFC            # -Inf
    b[9, 200] = 0x7C           # +Inf and -Inf in one column: NaN
    b[20, 64] = 0x7D           # NaN
    a[:, 500] = 0x00
    b[30, 500] = 0x7C          # Inf x 0: NaN
    assert_bits_equal(gpu_run(cs, a, b), oracle_full(cs, a, b), f"t7 fast={fast} S={S}")
print("ok")
'''


@pytest.mark.parametrize("tile", TILES)
def test_forced_tile_is_bit_exact(tile):
    import __graft_entry__
    __graft_entry__.build()
    name, _, extra = tile.partition(":")
    env = dict(os.environ, EMU_FP8_TILE=name)
    env.pop("EMU_FP8_TC", None)
    if extra == "TC":
        env["EMU_FP8_TC"] = "1"
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]
