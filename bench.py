"""Benchmark of the emulated FP8 scaled GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--shard replicas|columns]

One step = one emu_scaled_mm call over one batch of synthetic inputs already
resident in HBM: decode, block-aligned truncating accumulation, split combine and
epilogue (every step of the hot path).  The default workload is the projection
batch, the largest single-GPU workload (M=8192 tokens, K=1920, N=5760, E4M3 x E4M3,
bf16 output, fast accumulation, S=1, hopper preset).  The metric is emulated
TFLOP/s = 2*M*N*K / time.

Timing: W untimed warm-up steps; then K steps, each preceded by an untimed L2
flush (a 256 MiB write, larger than the 129 MB L2) and bracketed by CUDA events on
the launching stream; barrier + synchronize on both sides of the timed region; the
maximum over ranks.  SM clocks and throttle reasons are sampled through NVML every
10 ms during the timed region (nvidia-smi every 200 ms when NVML cannot be loaded).

Roofline: the denominators are measured in the same run by libemupeaks (the
instruction rates of the pipes the kernel issues on, lane-operations per clock per
SM) times the SM count and the maximum SM clock.  The headline fraction is against
the rate at which the GB300 runs the GEMM's own inner loop on a 4 x 4 thread tile
(per output and k-pair 1.5 packed f32x2 instructions and 0.5 DPX add-max per MAC,
operands loaded from shared memory, every operand a per-thread register); beside it
the same arithmetic with operands shared by all threads (a register-file-light
upper bound), the FP32 pipe alone, the algorithmic count of 5 integer
lane-operations per MAC against the measured integer peak, and for the split-K
shapes the HBM bytes against the measured HBM bandwidth and the serial-chain
latency per block.

CPU baseline and parity: the CPU oracle (exact integer arithmetic, every host
thread) is timed on stripes of the same workload -- a 64-row stripe, then column
slabs -- and every output it produces is compared bit for bit with the timed GPU
output; the line carries "parity": {"checked", "mismatches"}, and the run fails
on any mismatch.

e2e: the same metric through the host-buffer call (scaled_mm_host): every step uploads
its pinned host operands and copies its result back, inside the timed region; steps
alternate between two streams and two staging buffers, so one step's upload runs under
the previous step's GEMM.

N > 1 (torchrun): --shard replicas (default): every rank runs the whole workload on
its own GPU (the GEMM has no exchange step; weak scaling); --shard columns: the
ranks split N into column slabs of the one workload (strong scaling, no data-path
collective).  value = all ranks' flops / the maximum time over ranks.

--impl reference runs the CPU oracle (the slow, exact reference model) on the host
cores on a bounded sample of the same workload, rank 0 only.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_exact_fp8_gb300 import workloads as W  # noqa: E402

METRIC = "emulated FP8 GEMM TFLOP/s (2MNK/s) bit-exact vs oracle; % of INT-ALU/HBM roofline"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "projection-N5760"
OPS_PER_MAC = 5             # algorithmic: exponent add, max, significand multiply, align shift, add
FP32_OPS_PER_MAC = 3        # the kernel's exact product, truncating multiply and exact add


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return None


KERNEL_SOURCES = ("bit_exact_fp8_gb300/csrc/emu_kernels.cuh", "bit_exact_fp8_gb300/csrc/emu_tc.cuh",
                  "bit_exact_fp8_gb300/csrc/emu_api.cu")


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: comments and blank space do not count, so a
    comment edit keeps a profile summary valid and any code change invalidates it."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)     # block comments
        src = re.sub(r"//[^\n]*", " ", src)                   # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def profile_summary(workload: str):
    """The committed ncu summary of this workload's GEMM launch (profiles/<kernel>_<workload>.md,
    the kernel emu_gemm, emu_chain, emu_wsp, or emu_wst for the W tile with tensor-core
    products, which runs only with EMU_FP8_TC=1), if it was taken on the current kernel
    sources: {"traffic": DRAM bytes per launch, "ncu": {...}}."""
    import glob
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", f"emu_*_{workload}.md")))
    tc = os.environ.get("EMU_FP8_TC") == "1"
    wst = [p for p in paths if os.path.basename(p).startswith("emu_wst_")]
    paths = wst if (tc and wst) else [p for p in paths if p not in wst]
    if not paths:
        return None
    for path in paths:
        got = _profile_fields(path)
        if got is not None:
            return got
    return None


def _profile_fields(path: str):
    fields, table = {}, {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
            elif line.startswith("| ") and line.count("|") == 3:
                k, v = [x.strip() for x in line.strip().strip("|").split("|")]
                table[k] = v
    if fields.get("kernel source sha256") != kernel_source_hash():
        return None

    def num(key):
        try:
            return float(table[key].split()[0])
        except (KeyError, ValueError, IndexError):
            return None
    try:
        traffic = float(fields["dram bytes per launch"])
    except (KeyError, ValueError):
        traffic = None
    return {"traffic": traffic,
            "ncu": {"source": os.path.relpath(path, ROOT),
                    "issue_active_pct": num("smsp__issue_active.avg.pct_of_peak_sustained_active"),
                    "fma_pipe_pct": num("sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active"),
                    "alu_pipe_pct": num("sm__pipe_alu_cycles_active.avg.pct_of_peak_sustained_active"),
                    "shared_pipe_pct": num("l1tex__data_pipe_lsu_wavefronts_mem_shared.sum.pct_of_peak_sustained_elapsed")}}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# clocks during the timed region
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class Clocks:
    """SM clock, power and throttle reasons of one GPU, sampled every 10 ms through
    NVML (libnvidia-ml, read-only queries) from a host thread; falls back to
    nvidia-smi every 200 ms when NVML cannot be loaded."""

    def __init__(self, dev: torch.device):
        self.dev = dev
        self.samples = []
        self.nvml = None
        self.handle = None
        self.proc = None
        self._stop = threading.Event()
        try:
            self._open_nvml()
        except (OSError, AttributeError):
            self.nvml = None

    def _open_nvml(self):
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.dev)
        ok = False
        if all(hasattr(props, k) for k in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
            for fmt in ("{:08x}:{:02x}:{:02x}.0", "{:04x}:{:02x}:{:02x}.0"):
                bus = fmt.format(props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
                if L.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0:
                    ok = True
                    break
        if not ok and hasattr(props, "uuid"):
            uid = ("GPU-" + str(props.uuid)).encode()
            ok = L.nvmlDeviceGetHandleByUUID(uid, ctypes.byref(h)) == 0
        if not ok:
            raise OSError("no NVML handle for the CUDA device")
        self.nvml, self.handle = L, h
        self.reason_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(L, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None

    def _poll(self):
        L, h = self.nvml, self.handle
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                p = pw.value / 1e3 if L.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                r = rs.value if self.reason_fn(h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), p, int(r)))
            self._stop.wait(0.010)

    def start(self):
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.out = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev.index or 0),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            self._stop.set()
            self.thread.join(timeout=5)
            sm = [s[0] for s in self.samples]
            reasons = sorted({name for _, _, r in self.samples for bit, name in _REASONS.items()
                              if r & bit})
            pw = [s[1] for s in self.samples if s[1] is not None]
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "samples": len(sm), "sampler": "nvml 10 ms",
                    "power_w_max": max(pw) if pw else None, "reasons": reasons}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                    "reasons": ["no clock sampler available"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.out) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[3:7]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.out)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "sampler": "nvidia-smi 200 ms", "reasons": sorted(reasons)}


def torch_fp8(fmt):
    return torch.float8_e4m3fn if fmt == "e4m3fn" else torch.float8_e5m2


def out_torch_dtype(od):
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[od]


def out_bits(y: torch.Tensor) -> np.ndarray:
    y = y.cpu()
    if y.dtype == torch.float32:
        return y.view(torch.int32).numpy().view(np.uint32)
    return y.view(torch.int16).numpy().view(np.uint16)


def config_dict(cs, l2_note):
    return {"workload": f"{cs.name}: M={cs.M} N={cs.N} K={cs.K} {cs.fmt_a} x {cs.fmt_b} "
                        f"-> {cs.out_dtype}, {'fast' if cs.fast_accum else 'slow'} accumulation, "
                        f"S={cs.split_S}, {cs.preset} preset",
            "M": cs.M, "N": cs.N, "K": cs.K, "fmt_a": cs.fmt_a, "fmt_b": cs.fmt_b,
            "out_dtype": cs.out_dtype, "fast_accum": cs.fast_accum, "split_S": cs.split_S,
            "preset": cs.preset, "l2": l2_note}


def dtype_label(cs):
    return f"{cs.fmt_a}x{cs.fmt_b}->{cs.out_dtype}"


def blocks_per_chain(cs):
    """32- or 16-product blocks in one split's chain (the longest split)."""
    B = 32 if cs.preset == "hopper" else 16
    kt = 128 if cs.preset == "hopper" else 64
    T = -(-cs.K // kt)
    per_split = -(-T // cs.split_S) * kt
    return -(-min(cs.K, per_split) // B)


# ---------------------------------------------------------------------------
def oracle_leg(cs, a, b, budget_s: float, got=None):
    """The CPU oracle as it stands, on every host thread, timed on stripes of the
    workload until about budget_s seconds of work: a 64-row stripe first (every
    output of a workload with M <= 64), then column slabs at rotating offsets.
    When ``got`` (the timed GPU output's bits) is given, every output the oracle
    produces is compared with it.  Returns (TFLOP/s, cores, sample, parity)."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    t_total, macs_total, checked, bad = 0.0, 0, 0, 0
    first_bad = []
    seen = np.zeros((cs.M, cs.N), dtype=bool) if got is not None else None

    def run(a_part, b_part, rows, cols):
        nonlocal t_total, macs_total, checked, bad
        t0 = time.perf_counter()
        want = oracle.scaled_mm(a_part, b_part, cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b,
                                cs.out_dtype, cs.fast_accum, cs.split_S, cs.preset,
                                nthreads=cores)
        dt = time.perf_counter() - t0
        t_total += dt
        macs_total += a_part.shape[0] * b_part.shape[0] * a_part.shape[1]
        if got is not None:
            g = got[rows, cols]
            diff = np.flatnonzero(g.ravel() != want.ravel())
            checked += want.size
            bad += diff.size
            seen[rows, cols] = True
            if diff.size and len(first_bad) < 5:
                first_bad.append(f"rows {rows.start}.. cols {cols.start}..: {diff.size} differ")
        return dt

    rng = np.random.default_rng(2024)
    r0 = int(rng.integers(0, max(1, cs.M - 64 + 1)))
    rows = slice(r0, min(cs.M, r0 + 64))
    run(a[rows], b, rows, slice(0, cs.N))
    pieces = 1
    ncols, c0 = 16, int(rng.integers(0, max(1, cs.N // 16))) * 16
    while t_total < budget_s:
        cols = slice(c0, min(cs.N, c0 + ncols))
        dt = run(a, b[cols], slice(0, cs.M), cols)
        pieces += 1
        c0 = (c0 + 7 * 16 + ncols) % max(16, cs.N - ncols + 1) // 16 * 16
        if dt < budget_s / 20:
            ncols = min(cs.N, ncols * 2)
    sample = (f"{pieces} oracle calls on stripes of the {cs.name} workload (a 64-row stripe, "
              f"then column slabs; {macs_total / 1e9:.2f} GMAC, {t_total:.1f} s, all {cores} "
              "host threads)")
    parity = None
    if got is not None:
        parity = {"checked": int(checked), "mismatches": int(bad),
                  "distinct_outputs": int(seen.sum()), "of_outputs": int(cs.M * cs.N),
                  "what": "every output the CPU-baseline oracle calls produce, bit for bit "
                          "against the timed GPU output"}
        if first_bad:
            parity["first"] = first_bad
    return 2.0 * macs_total / t_total / 1e12, cores, sample, parity


def run_reference(args, cs):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    a, b = W.make_inputs(cs)
    steps, warmup = args.steps, args.warmup
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    # bounded per-step sample: a column slice sized so that the whole run takes ~60 s
    t0 = time.perf_counter()
    oracle.scaled_mm(a, b[:16], cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b, cs.out_dtype,
                     cs.fast_accum, cs.split_S, cs.preset, nthreads=cores)
    per_col = max(1e-6, (time.perf_counter() - t0) / 16)
    cols = int(max(1, min(cs.N, 60.0 / (steps + warmup) / per_col)))
    macs_step = cs.M * cols * cs.K
    times = []
    for i in range(warmup + steps):
        c0 = (i * cols) % max(1, cs.N - cols + 1)
        t0 = time.perf_counter()
        oracle.scaled_mm(a, b[c0:c0 + cols], cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b,
                         cs.out_dtype, cs.fast_accum, cs.split_S, cs.preset, nthreads=cores)
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = 2.0 * macs_step * steps / total / 1e12
    sample = f"each step: {cs.M} x {cols} outputs of the {cs.name} workload (K={cs.K})"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": steps, "warmup": warmup, "ms_per_step": 1e3 * total / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "config": config_dict(cs, "host CPU, no GPU"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def roofline(cs, t_step, rates, peaks, sms, prof):
    """The roofline object of the GEMM kernel (see the module docstring)."""
    mhz = (peaks or {}).get("sm_max_mhz", 2070.0)
    clk = sms * mhz * 1e6
    macs = cs.M * cs.N * cs.K
    tflops = 2.0 * macs / t_step / 1e12
    mix = rates["emulation_mix_macs"]
    vec = rates.get("emulation_mix_vector_macs")
    tile = rates.get("emulation_tile_macs")
    packed = min(rates[k] for k in ("f32x2_fmul_rz_subnormal", "f32x2_fmul_rn_normal",
                                    "f32x2_fadd_subnormal"))
    int_peak = max(rates[k] for k in ("imad", "iadd3", "lop3", "prmt", "dpx_viaddmax_s16x2",
                                      "imad_iadd3_mixed"))
    roof_macs = tile if tile else mix
    peak = 2.0 * roof_macs * clk / 1e12
    roof = {"bound": "alu", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
            "frac": tflops / peak,
            "traffic": prof["traffic"] if prof else None,
            "note": (f"peak = measured rate of the GEMM's inner loop on a 4 x 4 thread tile "
                     f"(per output and k-pair: packed exact product, truncating multiply and add, "
                     f"and a DPX add-max; operands loaded from a decoded stage in shared memory; "
                     f"no decode, scale or barrier): {roof_macs:.1f} MAC/clk/SM, libemupeaks in "
                     f"this run, x {sms} SMs x {mhz:.0f} MHz (sm_max_mhz); achieved = 2MNK / "
                     f"event time. The same arithmetic issues at {mix:.1f} MAC/clk/SM when its "
                     f"second operands are the same in every thread"
                     + (f", and at {vec:.1f} with per-thread operands and little reuse" if vec else "")
                     + ": register-file reads, not the FP32 pipe, bound it")}
    roof["uniform_operand_mix"] = {"macs_per_clk_sm": mix, "peak": 2.0 * mix * clk / 1e12,
                                   "frac": tflops / (2.0 * mix * clk / 1e12)}
    roof["fp32_pipe"] = {"ops_per_mac": FP32_OPS_PER_MAC, "unit": "Tops/s",
                         "achieved": FP32_OPS_PER_MAC * macs / t_step / 1e12,
                         "peak": packed * clk / 1e12,
                         "peak_lane_ops_per_clk_sm": packed,
                         "frac": FP32_OPS_PER_MAC * macs / t_step / (packed * clk)}
    roof["algorithmic"] = {"ops_per_mac": OPS_PER_MAC, "unit": "Tops/s",
                           "achieved": OPS_PER_MAC * macs / t_step / 1e12,
                           "peak": int_peak * clk / 1e12,
                           "peak_lane_ops_per_clk_sm": int_peak,
                           "frac": OPS_PER_MAC * macs / t_step / (int_peak * clk),
                           "note": "5 integer lane-ops per MAC against the measured 32-bit integer "
                                   "issue peak; the kernel does the work on the FP32 pipe, so "
                                   "this fraction can exceed 1"}
    roof["measured_issue_rates"] = {k: round(v, 2) for k, v in rates.items()}
    if prof:
        roof["ncu"] = prof["ncu"]
    if peaks and "hbm_gbs" in peaks:
        esz = 4 if cs.out_dtype == "f32" else 2
        byts = cs.M * cs.K + cs.N * cs.K + cs.M * cs.N * esz
        if cs.split_S > 1:
            byts += 2 * cs.split_S * cs.M * cs.N * 4        # partials written and read back
        roof["hbm"] = {"bytes_per_step": byts, "achieved_gbs": byts / t_step / 1e9,
                       "peak_gbs": peaks["hbm_gbs"],
                       "frac": byts / t_step / 1e9 / peaks["hbm_gbs"],
                       "note": "algorithmic bytes (operands once, output, split partials) against "
                               "the measured copy bandwidth of MEASURED_PEAKS.json"}
    if cs.split_S > 1:
        nb = blocks_per_chain(cs)
        roof["latency"] = {"blocks_per_chain": nb,
                           "sm_clocks_per_block": t_step * mhz * 1e6 / nb,
                           "note": "serial blocks of one split's chain; clocks per block = step "
                                   "time x max SM clock / blocks (combine kernel included)"}
    return roof


def run_gpu(args, cs):
    from bit_exact_fp8_gb300 import _lib, api, peaks as peaks_mod
    from bit_exact_fp8_gb300.sharding import column_slab
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    a, b = W.make_inputs(cs)
    # column slabs: this rank's [n0, n1) of the one workload; replicas: all of it
    n0, n1 = (column_slab(cs.N, rank, ws) if (ws > 1 and args.shard == "columns")
              else (0, cs.N))
    Nl = n1 - n0
    A = torch.from_numpy(a).to(dev).view(torch_fp8(cs.fmt_a))
    Bt = torch.from_numpy(np.ascontiguousarray(b[n0:n1])).to(dev).view(torch_fp8(cs.fmt_b))
    sa = torch.tensor(cs.scale_a, dtype=torch.float32, device=dev)
    sb = torch.tensor(cs.scale_b, dtype=torch.float32, device=dev)
    od = out_torch_dtype(cs.out_dtype)
    out = torch.empty((cs.M, Nl), dtype=od, device=dev)
    need = api.workspace_bytes(cs.M, Nl, cs.split_S)
    wsbuf = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    P = api.preset_params(cs.preset)
    stream = torch.cuda.current_stream(dev)
    fmt = {"e4m3fn": _lib.EMU_E4M3FN, "e5m2": _lib.EMU_E5M2}
    odc = {"f32": _lib.EMU_OUT_F32, "bf16": _lib.EMU_OUT_BF16, "f16": _lib.EMU_OUT_F16}

    def step():
        if Nl == 0:
            return
        st = _lib.emu_scaled_mm(A.data_ptr(), fmt[cs.fmt_a], Bt.data_ptr(), fmt[cs.fmt_b],
                                cs.M, Nl, cs.K, sa.data_ptr(), sb.data_ptr(), out.data_ptr(),
                                odc[cs.out_dtype], int(cs.fast_accum), cs.split_S, P,
                                wsbuf.data_ptr(), wsbuf.numel(), stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"emu_scaled_mm failed: {st} {_lib.emu_last_error()}")

    launches_per_step = (1 + (1 if cs.split_S > 1 else 0)) if Nl else 0
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(dev)
    # the roofline's denominators, measured on this GPU before the timed region
    rates = peaks_mod.issue_rates()
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = Clocks(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    t_sum = sum(kernel_ms) / 1e3
    if ws > 1:
        from bit_exact_fp8_gb300.sharding import max_over_ranks
        t_sum = max_over_ranks(t_sum)
    got = out_bits(out) if (rank == 0 and Nl == cs.N) else None

    flops_step = 2.0 * cs.M * cs.N * cs.K
    job_flops = flops_step * (ws if args.shard == "replicas" else 1)
    value = job_flops * args.steps / t_sum / 1e12
    ms_step = 1e3 * t_sum / args.steps

    # roofline of the dominant kernel (the GEMM; for S > 1 the step also holds the
    # small combine kernel), on this rank's share of the work
    mine = W.shrink(cs, cs.M, Nl, cs.K) if Nl != cs.N else cs
    prof = profile_summary(args.workload) if (args.traffic is None and Nl == cs.N) else None
    if args.traffic is not None:
        prof = {"traffic": args.traffic, "ncu": {"source": "--traffic"}}
    roof = roofline(mine, t_sum / args.steps, rates, measured_peaks(),
                    torch.cuda.get_device_properties(dev).multi_processor_count, prof)

    # end to end through the public API's host-buffer call: every step uploads its
    # pinned host operands, computes and copies its result back into pinned host
    # memory, all inside the timed region.  Steps alternate between two streams and
    # two staging buffers, so step i + 1's upload runs under step i's GEMM (a stream
    # of calls, as a server would issue them); the region spans the first upload to
    # the last copy back.
    e2e = None
    if Nl and args.e2e_steps > 0:
        e2e_steps = max(3, min(args.steps, args.e2e_steps))
        a_h = torch.from_numpy(a).view(torch_fp8(cs.fmt_a)).pin_memory()
        b_h = torch.from_numpy(np.ascontiguousarray(b[n0:n1])).view(torch_fp8(cs.fmt_b)).pin_memory()
        lanes = 2
        e2e_streams = [torch.cuda.Stream(dev) for _ in range(lanes)]
        y_h = [torch.empty((cs.M, Nl), dtype=od).pin_memory() for _ in range(lanes)]
        stagings = [torch.empty(api.staging_bytes(cs.M, Nl, cs.K, cs.split_S, od),
                                dtype=torch.uint8, device=dev) for _ in range(lanes)]

        def e2e_call(i):
            with torch.cuda.stream(e2e_streams[i % lanes]):
                api.scaled_mm_host(a_h, b_h.t(), cs.scale_a, cs.scale_b, out_dtype=od,
                                   use_fast_accum=cs.fast_accum, splitk=cs.split_S,
                                   preset=cs.preset, out=y_h[i % lanes], staging=stagings[i % lanes],
                                   chunks=args.e2e_chunks, device=dev, synchronize=False)

        for i in range(2 * lanes):                       # warm-up (streams, pools, pages)
            e2e_call(i)
        torch.cuda.synchronize(dev)
        if ws > 1:
            dist.barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(e2e_streams[0])
        e2e_streams[1].wait_stream(e2e_streams[0])
        for i in range(e2e_steps):
            e2e_call(i)
        e2e_streams[0].wait_stream(e2e_streams[1])
        t1.record(e2e_streams[0])
        torch.cuda.synchronize(dev)
        t_e2e = t0.elapsed_time(t1) / 1e3
        if ws > 1:
            from bit_exact_fp8_gb300.sharding import max_over_ranks
            t_e2e = max_over_ranks(t_e2e)
        e2e = {"value": job_flops * e2e_steps / t_e2e / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": a.nbytes + Nl * cs.K,
               "d2h_bytes_per_step": cs.M * Nl * y_h[0].element_size(), "steps": e2e_steps,
               "chunks": args.e2e_chunks, "pipelined_streams": lanes,
               "api": "scaled_mm_host (emu_scaled_mm_host)"}

    cpu, parity = None, None
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, sample, parity = oracle_leg(cs, a, b, args.cpu_seconds, got)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        config = config_dict(cs, "flushed between timed steps (256 MiB write)")
        config["tile"] = api.tile_for(cs.M, Nl or cs.N, cs.K, use_fast_accum=cs.fast_accum,
                                      splitk=cs.split_S, preset=cs.preset)
        if ws > 1:
            config["parallelism"] = (f"{ws} replicas" if args.shard == "replicas"
                                     else f"{ws} column slabs of N")
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak" if args.shard == "replicas" else "strong",
                "vs_baseline": None, "dtype": dtype_label(cs),
                "data": "synthetic",
                "config": config,
                "roofline": roof, "cpu_baseline": cpu, "parity": parity, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clk, "wall_s_timed_region": wall}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    if parity is not None and parity["mismatches"]:
        sys.exit(f"parity: {parity['mismatches']} of {parity['checked']} outputs differ from the oracle")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="a workload case by name, or NAME@MxNxK: its recipe at those sizes")
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--shard", default="replicas", choices=("replicas", "columns"),
                    help="N > 1: whole workload per rank (weak) or column slabs of it (strong)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--e2e-chunks", type=int, default=1,
                    help="column slabs of the host-buffer call (copies overlap the GEMM)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the GEMM kernel from an ncu capture")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle leg (and with it the parity check)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cs = W.named(args.workload)
    if args.impl == "reference":
        run_reference(args, cs)
    else:
        run_gpu(args, cs)


if __name__ == "__main__":
    main()
