"""Benchmark of the emulated FP8 scaled GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one emu_scaled_mm call over one batch of synthetic inputs already
resident in HBM: decode, block-aligned truncating accumulation, split combine and
epilogue (every step of the hot path).  The default workload is the linear-layer
shape of the documentation's example (M=64, K=1920, N=5760, E4M3 x E4M3, bf16
output, fast accumulation, S=1, hopper preset).  The metric is emulated TFLOP/s =
2*M*N*K / time.

Timing: W untimed warm-up steps; then K steps, each preceded by an untimed L2
flush (a 256 MiB write, larger than the 129 MB L2) and bracketed by CUDA events on
the launching stream; barrier + synchronize on both sides of the timed region; the
maximum over ranks.  Clocks are sampled with nvidia-smi during the timed region.

e2e: the same metric through the host-buffer call (scaled_mm_host): every step uploads
its pinned host operands and copies its result back, inside the timed region; steps
alternate between two streams and two staging buffers, so one step's upload runs under
the previous step's GEMM.

N > 1 (torchrun): every rank runs the same workload on its own GPU (the GEMM has no
exchange step: replicas, weak scaling); value = all ranks' flops / max time.

--impl reference runs the CPU oracle (the slow, exact reference model) on the host
cores on a bounded sample of the same workload, rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_exact_fp8_gb300 import workloads as W  # noqa: E402

METRIC = "emulated FP8 GEMM TFLOP/s (2MNK/s) bit-exact vs oracle; % of INT-ALU/HBM roofline"
UNIT = "TFLOP/s"
SMS = 152
LANES_PER_SM = 128          # 4 sub-partitions x 32 lanes: one warp instruction per clock each
OPS_PER_MAC = 5             # exponent add, max, significand multiply, align shift, add
FP32_OPS_PER_MAC = 3        # the kernel's exact product, truncating multiply and exact add


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return None


KERNEL_SOURCES = ("bit_exact_fp8_gb300/csrc/emu_kernels.cuh", "bit_exact_fp8_gb300/csrc/emu_api.cu")


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


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary of
    this workload, if it was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"emu_gemm_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel source sha256") != kernel_source_hash():
        return None
    try:
        return float(fields["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


def alu_peak_tops(peaks):
    """Issue-slot peak of 32-bit lane operations: SMs x 128 lanes x max SM clock."""
    mhz = (peaks or {}).get("sm_max_mhz", 2070.0)
    return SMS * LANES_PER_SM * mhz * 1e6 / 1e12, mhz


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.out = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
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
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.out)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def torch_fp8(fmt):
    return torch.float8_e4m3fn if fmt == "e4m3fn" else torch.float8_e5m2


def out_torch_dtype(od):
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[od]


def config_dict(cs, l2_note):
    return {"workload": f"{cs.name}: M={cs.M} N={cs.N} K={cs.K} {cs.fmt_a} x {cs.fmt_b} "
                        f"-> {cs.out_dtype}, {'fast' if cs.fast_accum else 'slow'} accumulation, "
                        f"S={cs.split_S}, {cs.preset} preset",
            "M": cs.M, "N": cs.N, "K": cs.K, "fmt_a": cs.fmt_a, "fmt_b": cs.fmt_b,
            "out_dtype": cs.out_dtype, "fast_accum": cs.fast_accum, "split_S": cs.split_S,
            "preset": cs.preset, "l2": l2_note}


# ---------------------------------------------------------------------------
def oracle_rate(cs, a, b, budget_s: float):
    """Time the CPU oracle (as it stands) on column slices of the workload until
    about budget_s seconds of work; returns (TFLOP/s, cores, sample description)."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    ncols = 16
    t_total, macs_total, reps = 0.0, 0, 0
    start_col = 0
    while t_total < budget_s:
        cols = slice(start_col, start_col + ncols)
        t0 = time.perf_counter()
        oracle.scaled_mm(a, b[cols], cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b, cs.out_dtype,
                         cs.fast_accum, cs.split_S, cs.preset, nthreads=cores)
        dt = time.perf_counter() - t0
        t_total += dt
        macs_total += a.shape[0] * ncols * a.shape[1]
        reps += 1
        start_col = (start_col + ncols) % max(1, b.shape[0] - ncols)
        if dt < budget_s / 20:
            ncols = min(b.shape[0], ncols * 2)
    sample = (f"{reps} oracle calls on column slices of the {cs.name} workload "
              f"({macs_total / 1e9:.2f} GMAC, {t_total:.1f} s, all {cores} host threads)")
    return 2.0 * macs_total / t_total / 1e12, cores, sample


def run_reference(args, cs):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    a, b = W.make_inputs(cs)
    steps, warmup = args.steps, args.warmup
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    # bounded per-step sample: a column slice sized so the whole run takes ~60 s
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
def run_gpu(args, cs):
    from bit_exact_fp8_gb300 import _lib, api
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    a, b = W.make_inputs(cs)
    A = torch.from_numpy(a).to(dev).view(torch_fp8(cs.fmt_a))
    Bt = torch.from_numpy(b).to(dev).view(torch_fp8(cs.fmt_b))
    sa = torch.tensor(cs.scale_a, dtype=torch.float32, device=dev)
    sb = torch.tensor(cs.scale_b, dtype=torch.float32, device=dev)
    od = out_torch_dtype(cs.out_dtype)
    out = torch.empty((cs.M, cs.N), dtype=od, device=dev)
    need = api.workspace_bytes(cs.M, cs.N, cs.split_S)
    wsbuf = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    P = api.preset_params(cs.preset)
    stream = torch.cuda.current_stream(dev)
    fmt = {"e4m3fn": _lib.EMU_E4M3FN, "e5m2": _lib.EMU_E5M2}
    odc = {"f32": _lib.EMU_OUT_F32, "bf16": _lib.EMU_OUT_BF16, "f16": _lib.EMU_OUT_F16}

    def step():
        st = _lib.emu_scaled_mm(A.data_ptr(), fmt[cs.fmt_a], Bt.data_ptr(), fmt[cs.fmt_b],
                                cs.M, cs.N, cs.K, sa.data_ptr(), sb.data_ptr(), out.data_ptr(),
                                odc[cs.out_dtype], int(cs.fast_accum), cs.split_S, P,
                                wsbuf.data_ptr(), wsbuf.numel(), stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"emu_scaled_mm failed: {st} {_lib.emu_last_error()}")

    launches_per_step = 1 + (1 if cs.split_S > 1 else 0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = Clocks(dev.index if ws == 1 else local)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)                      # let the sampler take a first reading
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if ws > 1:
        dist.barrier()
    clk = clocks.stop()
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    t_sum = sum(kernel_ms) / 1e3
    if ws > 1:
        from bit_exact_fp8_gb300.sharding import max_over_ranks
        t_sum = max_over_ranks(t_sum)

    flops_step = 2.0 * cs.M * cs.N * cs.K
    value = ws * flops_step * args.steps / t_sum / 1e12
    ms_step = 1e3 * t_sum / args.steps

    # roofline of the dominant kernel (the GEMM; for S > 1 the step also holds the
    # small combine kernel, so the GEMM's share is taken from the profile summary)
    peaks = measured_peaks()
    peak, mhz = alu_peak_tops(peaks)
    achieved = OPS_PER_MAC * cs.M * cs.N * cs.K / (t_sum / args.steps) / 1e12
    traffic = args.traffic if args.traffic is not None else profiled_traffic(args.workload)
    roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Tops/s",
            "frac": achieved / peak, "traffic": traffic,
            "note": f"{OPS_PER_MAC} lane-ops per MAC (algorithmic); peak = {SMS} SMs x "
                    f"{LANES_PER_SM} lanes x {mhz:.0f} MHz issue slots (recipe unit counts, "
                    "sm_max_mhz of MEASURED_PEAKS.json)"}
    # this implementation's own ceiling: pass 2 issues packed f32x2 instructions, so the
    # FP32 pipe (128 operations per clock per SM) bounds it at 3 FP32 operations per MAC
    roof["fp32_pipe"] = {"ops_per_mac": FP32_OPS_PER_MAC, "peak": peak,
                         "achieved": FP32_OPS_PER_MAC * achieved / OPS_PER_MAC,
                         "frac": FP32_OPS_PER_MAC * achieved / OPS_PER_MAC / peak}
    if peaks and "hbm_gbs" in peaks:
        bytes_step = cs.M * cs.K + cs.N * cs.K + cs.M * cs.N * (4 if cs.out_dtype == "f32" else 2)
        roof["hbm_gbs"] = bytes_step / (t_sum / args.steps) / 1e9
        roof["hbm_frac_of_measured"] = roof["hbm_gbs"] / peaks["hbm_gbs"]

    # end to end through the public API's host-buffer call: every step uploads its
    # pinned host operands, computes and copies its result back into pinned host
    # memory, all inside the timed region.  Steps alternate between two streams and
    # two staging buffers, so step i + 1's upload runs under step i's GEMM (a stream
    # of calls, as a server would issue them); the region spans the first upload to
    # the last copy back.
    e2e = None
    if rank == 0 or ws > 1:
        e2e_steps = max(3, min(args.steps, args.e2e_steps))
        a_h = torch.from_numpy(a).view(torch_fp8(cs.fmt_a)).pin_memory()
        b_h = torch.from_numpy(b).view(torch_fp8(cs.fmt_b)).pin_memory()
        lanes = 2
        e2e_streams = [torch.cuda.Stream(dev) for _ in range(lanes)]
        y_h = [torch.empty((cs.M, cs.N), dtype=od).pin_memory() for _ in range(lanes)]
        stagings = [torch.empty(api.staging_bytes(cs.M, cs.N, cs.K, cs.split_S, od),
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
        e2e = {"value": ws * flops_step * e2e_steps / t_e2e / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": a.nbytes + b.nbytes,
               "d2h_bytes_per_step": cs.M * cs.N * y_h[0].element_size(), "steps": e2e_steps,
               "chunks": args.e2e_chunks, "pipelined_streams": lanes,
               "api": "scaled_mm_host (emu_scaled_mm_host)"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, sample = oracle_rate(cs, a, b, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        config = config_dict(cs, "flushed between timed steps (256 MiB write)")
        config["tile"] = api.tile_for(cs.M, cs.N, cs.K, use_fast_accum=cs.fast_accum,
                                      splitk=cs.split_S, preset=cs.preset)
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": config,
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clk, "wall_s_timed_region": wall}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="linear")
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--e2e-chunks", type=int, default=1,
                    help="column slabs of the host-buffer call (copies overlap the GEMM)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the GEMM kernel from an ncu capture")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cs = W.case(args.workload)
    if args.impl == "reference":
        run_reference(args, cs)
    else:
        run_gpu(args, cs)


if __name__ == "__main__":
    main()
