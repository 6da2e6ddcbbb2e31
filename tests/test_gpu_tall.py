"""Tall problems: row tiles sit on grid.y, which holds at most 65535, so a problem
with more row tiles is launched in several parts, each starting at its row-tile
offset.  With the 4-row tile forced, M = 300000 needs 75000 row tiles (two
launches); sampled outputs, including rows beyond the first launch, must equal the
oracle's bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
import numpy as np
sys.path.insert(0, "tests")
from bit_exact_fp8_gb300 import workloads as W
from helpers import assert_bits_equal, gpu_run, oracle_sampled, sample_indices
for cs in (W.Case("tall-k4", 300000, 16, 64, out_dtype="bf16", fast_accum=True, seed=21),
           W.Case("tall-slow-f32", 270001, 32, 96, out_dtype="f32", fast_accum=False, seed=22)):
    a, b = W.make_inputs(cs)
    y = gpu_run(cs, a, b)
    im, jn = sample_indices(cs.M, cs.N, 200, seed=cs.seed)
    rows = np.array([65535 * 4 - 1, 65535 * 4, 65535 * 4 + 3, cs.M - 1], np.int64)
    im = np.concatenate([im, rows])
    jn = np.concatenate([jn, np.arange(len(rows)) % cs.N])
    assert_bits_equal(y[im, jn], oracle_sampled(cs, a, b, im, jn), cs.name)
print("ok")
'''


@pytest.mark.parametrize("tile", ["K4", "auto"])
def test_more_row_tiles_than_one_launch_holds(tile):
    import __graft_entry__
    __graft_entry__.build()
    env = dict(os.environ)
    if tile != "auto":
        env["EMU_FP8_TILE"] = tile
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]
