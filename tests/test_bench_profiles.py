"""The committed ncu summaries that bench.py reads for its roofline's DRAM traffic: each
parses, names its kernel and workload, and the bench takes the W kernel with tensor-core
products' summary only when that path is switched on (EMU_FP8_TC=1)."""
import glob
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_summary_parses():
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", "emu_*_*.md")))
    assert paths
    for path in paths:
        text = open(path).read()
        assert re.search(r"kernel source sha256: `[0-9a-f]{16}`", text), path
        assert re.search(r"dram bytes per launch: \d+", text), path
        assert "ncu --" in text and "--clock-control none" in text, path


def test_the_tensor_core_summary_only_with_the_switch(monkeypatch):
    monkeypatch.delenv("EMU_FP8_TC", raising=False)
    got = bench.profile_summary("projection-N5760")
    if got is not None:                          # current sources: the register-file W kernel
        assert os.path.basename(got["ncu"]["source"]).startswith("emu_wsp_")
    monkeypatch.setenv("EMU_FP8_TC", "1")
    got = bench.profile_summary("projection-N5760")
    if got is not None:
        assert os.path.basename(got["ncu"]["source"]).startswith("emu_wst_")
    # a workload without a tensor-core summary keeps its own
    got = bench.profile_summary("linear")
    if got is not None:
        assert os.path.basename(got["ncu"]["source"]).startswith("emu_gemm_")
