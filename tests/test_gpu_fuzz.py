"""Seeded randomized parity: shapes (ragged in M, N and K), format pairs, presets,
fast and slow accumulation, split factors, combine rules, output dtypes with and
without scale_result, the two input generators, and the tile (the chooser's pick
or a forced one) drawn at random.  Every output is compared bit for bit with the
oracle, the tolerance of every parity test here.  The draw is fixed by its seed,
so a failure reproduces."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# "W:TC": the W tile with tensor-core products (opt-in, EMU_FP8_TC=1)
TILES = ["auto", "M40", "M32", "M64", "S", "K8", "K4", "K8H", "K4H", "C2", "C4", "C1", "C1L", "W", "W:TC"]

CHILD = r'''
import sys
import numpy as np
sys.path.insert(0, "tests")
from bit_exact_fp8_gb300 import workloads as W
from helpers import assert_bits_equal, gpu_run, oracle_full
seed, count = int(sys.argv[1]), int(sys.argv[2])
wide = len(sys.argv) > 3 and sys.argv[3] == "wide"     # several CTAs of the large tiles
rng = np.random.default_rng(seed)
pairs = [("e4m3fn", "e4m3fn"), ("e4m3fn", "e5m2"), ("e5m2", "e4m3fn")]
for i in range(count):
    fa, fb = pairs[rng.integers(3)]
    preset = ("hopper", "ada")[rng.integers(2)]
    out = ("f32", "bf16", "f16", "e4m3fn", "e5m2")[rng.integers(5)]
    if out == "e5m2" and fa == fb == "e4m3fn":
        out = "e4m3fn"                                   # refused by cuBLASLt
    sr = float(rng.choice([0.25, 3.0, -1.5])) if out in ("e4m3fn", "e5m2") and rng.integers(2) else None
    M = int(rng.integers(1, 400 if wide else 100))
    N = 16 * int(rng.integers(1, 25 if wide else 9))
    K = 16 * int(rng.integers(1, 80 if wide else 160))
    S = int(rng.choice([1, 1, 2, 3, 5]))
    cs = W.Case(f"fuzz{seed}-{i}", M, N, K, fa, fb, out, fast_accum=bool(rng.integers(2)),
                split_S=S, preset=preset, gen=("gauss", "mixed")[rng.integers(2)],
                seed=int(rng.integers(1 << 30)), scale_a=float(rng.choice([1 / 64, 0.5, 3.0])),
                scale_b=float(rng.choice([1 / 32, 1.0, -2.0])), scale_result=sr)
    a, b = W.make_inputs(cs)
    assert_bits_equal(gpu_run(cs, a, b), oracle_full(cs, a, b),
                      f"{cs.name} M={M} N={N} K={K} S={S} {fa}x{fb}->{out} {preset} "
                      f"fast={cs.fast_accum} sr={sr}")
print("ok")
'''


def _run(tile, seed, count, *extra_args):
    import __graft_entry__
    __graft_entry__.build()
    env = dict(os.environ)
    env.pop("EMU_FP8_TC", None)
    name, _, extra = tile.partition(":")
    if name != "auto":
        env["EMU_FP8_TILE"] = name
    if extra == "TC":
        env["EMU_FP8_TC"] = "1"
    r = subprocess.run([sys.executable, "-c", CHILD, str(seed), str(count), *extra_args], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]


@pytest.mark.parametrize("tile", TILES)
def test_random_cases_are_bit_exact(tile):
    _run(tile, 1000 + TILES.index(tile), 100)


# M up to 399 and N up to 384: several CTAs of every tile, ragged in both directions
@pytest.mark.parametrize("tile", TILES)
def test_random_wide_cases_are_bit_exact(tile):
    _run(tile, 2000 + TILES.index(tile), 12, "wide")
