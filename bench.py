#!/usr/bin/env python
"""Benchmark: GEMM TFLOP/s on the 8192^3 BF16 workload with the fused
bias + GELU epilogue (A row-major, B column-major, bf16 D), 1 GPU per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one tcg_gemm launch over the whole 8192^3 problem with inputs
resident in HBM (A+B = 256 MiB > the 129 MB L2, so no flush is needed).  The
timed region is bracketed by a barrier and a device synchronise on both sides
and timed with CUDA events on the launching stream; rank 0 prints one JSON line.
Under torchrun each rank runs an independent replica (weak scaling, no
collective on the data path); the reported time is the max over ranks.

--impl reference times the oracle (plain C, fp64, host cores) on bounded row
samples of the same workload, reported in the same unit.

--workload picks one of the other parity workloads (4096^3 beta*C, 512^3,
the ragged and skinny shapes, 8192^3 e4m3 / MXFP8 / NVFP4, the 16-expert
grouped MoE GEMM through tcg_gemm_grouped); those whose inputs fit in L2 are
timed one launch per event pair with a 512 MiB L2 flush in between.  The
roofline object is then against HBM bandwidth (GB/s) when the pages'
intensity 2MNK / (b (MK + KN + MN)) puts the shape below the ridge point.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s and % of GB300 dense tensor peak (8192³ BF16), 1 GPU"
UNIT = "TFLOP/s"
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--role-stats", action="store_true",
                    help="instead of the bench line: per-CTA time of each role (the kernel's cycle "
                         "accounting, TCG_STATS=1) over --steps launches of the workload")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD,
                    help="the metric's workload (default) or one of the parity workloads, "
                         "measured the same way for the per-workload roofline table")
    return ap.parse_args()


# Workloads: name -> (case factory name in inputs, flush L2 between launches).
# Inputs that do not exceed the 129 MB L2 by a wide margin are timed one launch
# at a time with a 512 MiB L2 flush between launches (outside the timed events).
DEFAULT_WORKLOAD = "gemm8192_bias_gelu"
WORKLOADS = {
    "gemm8192_bias_gelu": (lambda inputs: inputs.square_8192_gelu(), False),
    "gemm4096_beta1": (lambda inputs: inputs.square_4096_beta(), True),
    "gemm512_uniform": (lambda inputs: inputs.square_512(integer=False), True),
    "ragged_4095x3001x1537": (lambda inputs: inputs.ragged(0, 1), True),
    "ragged_tight_4095x3001x1537": (lambda inputs: inputs.ragged_tight(1), True),
    "skinny_16x8192x8192": (lambda inputs: inputs.ragged(1, 1), True),
    "skinny_8192x128x8192": (lambda inputs: inputs.ragged(2, 1), True),
    "gemm8192_e4m3_bias_relu": (lambda inputs: inputs.fp8_8192_relu(), True),
    "gemm8192_mxe4m3_bias_relu": (lambda inputs: inputs.mxfp8_8192_relu("e4m3"), True),
    "gemm8192_nvfp4_bias_relu": (lambda inputs: inputs.nvfp4_8192_relu(), True),
    # grouped GEMM: 16 MoE experts, 32768 routed rows, 4096 x 4096 weights (768 MiB of operands)
    "grouped_moe16_32768x4096x4096_bias_gelu": (lambda inputs: inputs.grouped_moe(), False),
}


def is_grouped(case):
    return hasattr(case, "problems")


def head(case):
    """The problem whose shared attributes (types, layouts, epilogue) describe the case."""
    return case.problems[0] if is_grouped(case) else case


def largest(case):
    """The problem the oracle samples rows from (the only one for a single GEMM)."""
    return max(case.problems, key=lambda p: p.M) if is_grouped(case) else case

def metric_name(workload):
    return METRIC if workload == DEFAULT_WORKLOAD else f"GEMM TFLOP/s ({workload}), 1 GPU"


_EB = {"bf16": 2, "f16": 2, "e4m3": 1, "e5m2": 1, "f32": 4, "nvfp4": 0.5, "mxfp4": 0.5}


def case_bytes(case):
    """Algorithmic bytes of one launch: A and B once, C once if beta != 0, D once, bias once
    (summed over the problems of a grouped GEMM)."""
    from tiled_tensor_core_persistent_gb300 import analysis
    if is_grouped(case):
        return sum(case_bytes(p) for p in case.problems)
    return analysis.gemm_bytes(case.M, case.N, case.K, _EB[case.ab_dtype], _EB[case.d_dtype],
                               _EB[case.c_dtype] if case.C is not None else 0,
                               _EB[case.bias_dtype] if case.bias is not None else 0)


def workload_config(case, flush):
    if is_grouped(case):
        h = head(case)
        cfg = workload_config(h, flush)
        epi = cfg["workload"].split("D = ")[1].rsplit(" (", 1)[0]
        ab = sum(t.numel() * t.element_size() for p in case.problems for t in (p.A, p.B))
        cfg.update(
            workload=f"grouped gemm, {len(case.problems)} problems M_g x {h.N} x {h.K} "
                     f"(M_g = {'/'.join(str(p.M) for p in case.problems)}) {h.ab_dtype}, A {h.opA}-major / "
                     f"B {h.opB}-major, per problem D = {epi} ({case.name})",
            M=sum(p.M for p in case.problems), N=h.N, K=h.K, problems=[[p.M, p.N, p.K] for p in case.problems])
        if not flush:
            cfg["l2"] = f"inputs larger than L2 (A+B {ab / 2**20:.0f} MiB > 129 MB), no flush"
        return cfg
    epi = []
    if case.C is not None:
        epi.append(f"beta*C ({case.c_dtype})")
    if case.bias is not None:
        epi.append(f"bias[N] ({case.bias_dtype})")
    if case.act != "none":
        epi.append(case.act + ("(erf)" if case.act == "gelu" else ""))
    ab = sum(t.numel() * t.element_size() for t in (case.A, case.B))
    return {"workload": f"gemm {case.M}x{case.N}x{case.K} {case.ab_dtype}, A {case.opA}-major / "
                        f"B {case.opB}-major, D = {' + '.join(['alpha*A@B'] + epi)} -> {case.d_dtype} "
                        f"({case.name}, seed {case.meta.get('seed')}, {case.meta.get('dist')})",
            "M": case.M, "N": case.N, "K": case.K, "ab_dtype": case.ab_dtype,
            "d_dtype": case.d_dtype, "epilogue": "+".join(epi) or "none", "accumulate": "f32",
            "l2": ("512 MiB L2 flush (write, then read back) between launches, outside the timed events" if flush else
                   f"inputs larger than L2 (A+B {ab / 2**20:.0f} MiB > 129 MB), no flush"),
            "parallelism": "replicas (one independent GEMM per GPU)"}


def launches_per_step(case, dc, tcg):
    """Kernel launches of one library call: the GEMM, plus the packing kernel
    when A or B is not TMA-addressable (the slow path sizes a larger workspace
    for the packed copies)."""
    if is_grouped(case) or case.K == 0 or dc.ab_dtype in ("mxe4m3", "mxe5m2", "nvfp4", "mxfp4"):
        return 1
    packs = tcg.workspace_size_for(case.M, case.N, case.K, dc.ab_dtype, dc.A, case.lda, case.opA, dc.B, case.ldb,
                                   case.opB) > tcg.workspace_size(case.M, case.N, case.K, dc.ab_dtype)
    return 2 if packs else 1


def cpu_model():
    """The host CPU's model name (lscpu), for the oracle's timings."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform_processor()


def platform_processor():
    import platform
    return platform.processor() or None


def run_env(device_index=None):
    """Versions and device of this run (recorded beside the numbers)."""
    import platform
    import torch
    env = {"python": platform.python_version(), "torch": torch.__version__, "cuda": torch.version.cuda,
           "host": platform.machine(), "host_cores": os.cpu_count(), "cpu_model": cpu_model()}
    if device_index is not None and torch.cuda.is_available():
        env["device"] = torch.cuda.get_device_name(device_index)
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(device_index), "--query-gpu=driver_version",
                                  "--format=csv,noheader"], capture_output=True, text=True, timeout=20)
            env["driver"] = out.stdout.strip() or None
        except Exception:
            env["driver"] = None
    return env


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"bf16_tflops": FALLBACK_PEAK_TFLOPS, "hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def _code_only(src):
    """C/C++ source without its comments and with its blank space collapsed
    (string and character literals kept as they are)."""
    out, i, n, quote = [], 0, len(src), None
    while i < n:
        c = src[i]
        if quote:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(src[i + 1])
                i += 2
                continue
            if c == quote:
                quote = None
            i += 1
        elif c in "\"'":
            quote = c
            out.append(c)
            i += 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash(csrc):
    """Hash of the code in directory `csrc`: every file except the test-only
    debug_* kernels (which take no part in a GEMM), without comments and blank
    space."""
    h = hashlib.sha256()
    for name in sorted(n for n in os.listdir(csrc) if not n.startswith("debug_")):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def kernel_source_hash():
    """Hash of the GEMM's code (source_hash of the package's csrc/): the
    recorded DRAM traffic stays valid across comment edits and lapses with any
    change to the code."""
    return source_hash(os.path.join(ROOT, "tiled_tensor_core_persistent_gb300", "csrc"))


def recorded_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(key)
        if e and e.get("kernel_source_hash") == kernel_source_hash():
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def max_over_ranks(pg, value, device):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def oracle_problem(case):
    import oracle
    from tiled_tensor_core_persistent_gb300 import inputs
    ab = {"bf16": oracle.BF16, "f16": oracle.F16, "e4m3": oracle.E4M3, "e5m2": oracle.E5M2,
          "nvfp4": oracle.E2M1, "mxfp4": oracle.E2M1}
    vec = {"bf16": oracle.BF16, "f32": oracle.F32}
    return oracle.Problem(
        case.M, case.N, case.K, inputs.raw_bits(case.A), case.lda,
        oracle.ROW if case.opA == "row" else oracle.COL,
        inputs.raw_bits(case.B), case.ldb, oracle.ROW if case.opB == "row" else oracle.COL,
        alpha=case.alpha, beta=case.beta, C=inputs.raw_bits(case.C), ldc=case.ldc,
        bias=inputs.raw_bits(case.bias), act=case.act, scale_a=case.scale_a, scale_b=case.scale_b,
        ab_dtype=ab[case.ab_dtype], c_dtype=vec[case.c_dtype] if case.C is not None else None,
        bias_dtype=vec[case.bias_dtype] if case.bias is not None else None,
        sfa=case.sfa, sfb=case.sfb, block=case.sf_block,
        sf_format=oracle.SF_UE4M3 if case.sf_format == "ue4m3" else oracle.SF_E8M0)


def cpu_oracle_rows(case, rows, nthreads=0, prob=None):
    import numpy as np
    prob = prob if prob is not None else oracle_problem(case)
    cols = np.arange(case.N, dtype=np.int32)
    t0 = time.perf_counter()
    prob.select(np.asarray(rows, dtype=np.int32), cols, nthreads)
    return time.perf_counter() - t0


def run_reference(args):
    """The oracle timed on host cores, bounded row samples per step."""
    world, rank, local, pg = dist_setup(args)
    if rank != 0:
        return 0
    from tiled_tensor_core_persistent_gb300 import inputs
    whole = WORKLOADS[args.workload][0](inputs)
    case = largest(whole)
    cores = os.cpu_count() or 1
    # size each step so the whole run stays within about a minute
    prob = oracle_problem(case)
    probe = cpu_oracle_rows(case, [0, 1], prob=prob)
    per_row = probe / 2
    budget_s = 60.0
    rows_per_step = max(1, int(budget_s / max(1, args.steps + args.warmup) / max(per_row, 1e-6)))
    rows_per_step = min(rows_per_step, 64)
    rng_rows = lambda i: [(i * rows_per_step + r) % case.M for r in range(rows_per_step)]
    for i in range(args.warmup):
        cpu_oracle_rows(case, rng_rows(i), prob=prob)
    t = 0.0
    for i in range(args.steps):
        t += cpu_oracle_rows(case, rng_rows(args.warmup + i), prob=prob)
    flops = 2.0 * rows_per_step * case.N * case.K * args.steps
    value = flops / t / 1e12
    sample = f"{rows_per_step} full rows of D (x {case.N} cols x K={case.K}) per step" + \
        (f", of the grouped GEMM's largest problem ({case.M} rows)" if is_grouped(whole) else "")
    line = {"impl": "reference", "metric": metric_name(args.workload), "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(whole, WORKLOADS[args.workload][1]),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "env": run_env()}
    print(json.dumps(line), flush=True)
    return 0


def timed_launches(args, dc, stream, device, flush):
    """Milliseconds of args.steps launches: back to back between two events, or
    (flush) one launch per event pair with an L2 flush outside each pair."""
    import torch
    if not flush:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            dc.run(stream)
        ev1.record(stream)
        torch.cuda.synchronize(device)
        return ev0.elapsed_time(ev1)
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i, (a, b) in enumerate(evs):
            # write 512 MiB, then read it back: L2 ends up holding clean lines
            # of the scrub buffer, so no write-back of the flush competes with
            # the timed launch for DRAM bandwidth
            scrub.fill_(i & 0xFF)
            scrub.view(torch.int32).sum()
            a.record(stream)
            dc.run(stream)
            b.record(stream)
    torch.cuda.synchronize(device)
    return sum(a.elapsed_time(b) for a, b in evs)


def launch_distribution(dc, stream, device, n):
    """Per-launch times (ms) of n launches, each between its own pair of events
    on the launching stream, back to back (outside the timed region): the
    median and the p10 / p90 spread of single launches."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            dc.run(stream)
            b.record(stream)
    torch.cuda.synchronize(device)
    ms = sorted(a.elapsed_time(b) for a, b in evs)
    pick = lambda q: ms[min(n - 1, int(q * (n - 1) + 0.5))]
    return {"median_ms": statistics.median(ms), "p10_ms": pick(0.1), "p90_ms": pick(0.9), "n": n,
            "how": "one event pair per launch, launches back to back, after the timed region"}


def run_ours(args):
    import torch
    world, rank, local, pg = dist_setup(args)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import tiled_tensor_core_persistent_gb300 as tcg
    from tiled_tensor_core_persistent_gb300 import _build, analysis, harness, inputs
    if rank == 0:
        _build.build()
    barrier(pg, device)
    tcg.lib()

    factory, flush = WORKLOADS[args.workload]
    case = factory(inputs)
    stream = torch.cuda.Stream(device=device)
    if is_grouped(case):
        dc = harness.GroupedDeviceCase(case, device=device, stream=stream)
    else:
        dc = harness.DeviceCase(case, device=device, stream=stream)
    torch.cuda.synchronize(device)

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            dc.run(stream)
    torch.cuda.synchronize(device)
    st = tcg.device_status(dc.workspace, stream)
    if st != 0:
        raise RuntimeError(f"device status {st}: {tcg.last_error()}")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(pg, device)
    torch.cuda.synchronize(device)
    elapsed_ms = timed_launches(args, dc, stream, device, flush)
    torch.cuda.synchronize(device)
    barrier(pg, device)
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(pg, elapsed_ms, device)
    st = tcg.device_status(dc.workspace, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region: {tcg.last_error()}")

    ms_per_step = elapsed_ms / args.steps
    launches = launch_distribution(dc, stream, device, min(100, max(args.steps, 10))) if rank == 0 else None
    flops = case.flops
    value = world * flops * args.steps / (elapsed_ms * 1e-3) / 1e12
    per_launch_tflops = flops / (ms_per_step * 1e-3) / 1e12

    # end to end through the public API: pinned host inputs -> device, GEMM, D -> pinned host
    if is_grouped(case):
        make_dc = lambda: harness.GroupedDeviceCase(case, device=device, stream=stream)
    else:
        make_dc = lambda: harness.DeviceCase(case, device=device, stream=stream)
    e2e = run_e2e(args, case, dc, stream, device, tcg, make_dc) if args.e2e_steps > 0 else None

    peaks, peak_kind = load_peaks()
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAK_TFLOPS))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    in_bytes = _EB[head(case).ab_dtype]
    # dense tensor peak of the operand type: fp8 = 2x bf16 (nominal 4.5 vs 2.25 PFLOP/s)
    # dense tensor peak of the operand type from the measured bf16 peak and the
    # nominal dense ratios of GB300: fp8 4.5 / 2.25 = 2, fp4 13.5 / 2.25 = 6
    ratio = 6.0 if in_bytes == 0.5 else (2.0 if in_bytes == 1 else 1.0)
    tensor_peak = bf16_peak * ratio
    nominal = 2250.0 * ratio
    alg_bytes = case_bytes(case)
    if is_grouped(case):
        # the pages' intensity 2MNK / (b (MK + KN + MN)) over the whole batch
        intensity = flops / (in_bytes * sum(p.M * p.K + p.K * p.N + p.M * p.N for p in case.problems))
    else:
        intensity = analysis.boundary_intensity(case.M, case.N, case.K, in_bytes)
    hbm_bound = intensity * hbm * 1e-3 < tensor_peak
    gbs = alg_bytes / (ms_per_step * 1e-3) / 1e9
    roof = {"bound": "hbm" if hbm_bound else "tensor",
            "achieved": gbs if hbm_bound else per_launch_tflops,
            "peak": hbm if hbm_bound else tensor_peak,
            "unit": "GB/s" if hbm_bound else "TFLOP/s",
            "frac": (gbs / hbm) if hbm_bound else (per_launch_tflops / tensor_peak),
            "traffic": recorded_traffic(args.workload),
            "peak_kind": (f"{peak_kind} copy bandwidth" if hbm_bound else
                          f"{peak_kind} bf16 burst (cuBLAS 8192^3)" + (f" x {ratio:g} for the operand type" if ratio != 1 else "")),
            "peak_sustained": None if hbm_bound else
            peaks.get("bf16_tflops_sustained", 0) * ratio or None,
            "frac_of_sustained": None if hbm_bound or not peaks.get("bf16_tflops_sustained") else
            per_launch_tflops / (peaks["bf16_tflops_sustained"] * ratio),
            "tflops": per_launch_tflops, "gbs": gbs,
            "frac_of_nominal_tensor": per_launch_tflops / nominal,
            "algorithmic": "2*M*N*K flop per launch; bytes = A + B + D (+ C, bias) once",
            "model": {"intensity_flop_per_byte": intensity,
                      "roofline_tflops": analysis.roofline(nominal, intensity, hbm * 1e-3),
                      "algorithmic_bytes": alg_bytes}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # a bounded sample: about 15 s of oracle work on the host cores
        big = largest(case)
        prob = oracle_problem(big)
        n_probe = min(16, big.M)
        t_probe = cpu_oracle_rows(big, list(range(0, big.M, max(1, big.M // n_probe)))[:n_probe], prob=prob)
        nrows = int(min(big.M, max(n_probe, 15.0 / max(t_probe / n_probe, 1e-6))))
        t = cpu_oracle_rows(big, list(range(0, big.M, max(1, big.M // nrows)))[:nrows], prob=prob)
        cpu = {"value": 2.0 * nrows * big.N * big.K / t / 1e12, "unit": UNIT,
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{nrows} full rows of D ({nrows}x{big.N}x{big.K}), {t:.1f} s wall" +
                         (f", of the grouped GEMM's largest problem ({big.M} rows)" if is_grouped(case) else "")}

    if is_grouped(case):
        plan = tcg.grouped_plan([dict(M=p.M, N=p.N, K=p.K) for p in case.problems], head(case).ab_dtype)
    else:
        plan = tcg.plan(case.M, case.N, case.K, dc.ab_dtype, case.opA, case.opB)
    if rank == 0:
        line = {"metric": metric_name(args.workload),
                "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": head(case).ab_dtype, "data": "synthetic",
                "config": dict(workload_config(case, flush), plan=plan),
                "roofline": roof, "cpu_baseline": cpu, "clocks": clocks, "e2e": e2e, "launch_ms": launches,
                "gpu_launches": args.steps * launches_per_step(case, dc, tcg), "env": run_env(local)}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def inputs_blocked(sf):
    from tiled_tensor_core_persistent_gb300 import inputs
    return inputs.mx_blocked_layout(sf)


def run_e2e(args, case, dc, stream, device, tcg, make_dc):
    """End to end through the public API: every step copies its inputs from
    pinned host memory to the device, runs the GEMM and copies D back to pinned
    host memory.  Steps are pipelined as a serving loop would run them: two
    device buffer sets, the host-to-device copies on one stream, the GEMMs on
    the launching stream and the device-to-host copies on a third, so step
    i + 1's inputs travel while step i computes; a buffer set is refilled only
    after its previous result has been copied out."""
    import torch
    sets = [dc, make_dc()]
    # pinned host inputs (one copy, read by every step) and one pinned host D per set
    host_in = []
    for p in (case.problems if is_grouped(case) else [case]):
        host_in.append([t.pin_memory() if t is not None else None for t in (p.A, p.B, p.bias, p.C)] +
                       [torch.from_numpy(inputs_blocked(x)).pin_memory() if x is not None else None
                        for x in (p.sfa, p.sfb)])

    def pairs(d):
        parts = d.parts if is_grouped(case) else [d]
        ins, outs = [], []
        for hs, part in zip(host_in, parts):
            devs = [part.A, part.B, part.bias, part.C, part.sfa, part.sfb]
            ins += [(h, dv) for h, dv in zip(hs, devs) if h is not None]
            outs.append((torch.empty(part.D_view.shape, dtype=part.D_view.dtype).pin_memory(), part.D_view))
        return ins, outs

    io = [pairs(d) for d in sets]
    h2d = sum(h.numel() * h.element_size() for h, _ in io[0][0])
    d2h = sum(h.numel() * h.element_size() for h, _ in io[0][1])
    # (one stream per direction: chunking the copies over 2, 4 or 8 streams was
    # measured no faster on GB300: 1.49, 1.51, 1.54, 1.61 ms per 8192^3 step)
    s_in = torch.cuda.Stream(device=device)
    s_out = torch.cuda.Stream(device=device)

    def copies(pairs, st, to_device):
        with torch.cuda.stream(st):
            for h, dv in pairs:
                if to_device:
                    dv.copy_(h, non_blocking=True)
                else:
                    h.copy_(dv, non_blocking=True)

    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def step(i):
        k = i & 1
        if started[k]:
            s_in.wait_event(out_done[k])          # set k's previous result has left the device
        started[k] = True
        copies(io[k][0], s_in, True)
        in_done[k].record(s_in)
        stream.wait_event(in_done[k])
        sets[k].run(stream)
        comp_done[k].record(stream)
        s_out.wait_event(comp_done[k])
        copies(io[k][1], s_out, False)
        out_done[k].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize(device)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    n = max(1, args.e2e_steps)
    ev0.record(s_in)
    for i in range(n):
        step(i)
    s_out.wait_event(in_done[(n - 1) & 1])
    s_out.wait_event(comp_done[(n - 1) & 1])
    ev1.record(s_out)
    torch.cuda.synchronize(device)
    ms = ev0.elapsed_time(ev1) / n
    for d in sets:
        st = tcg.device_status(d.workspace, stream)
        if st != 0:
            raise RuntimeError(f"device status {st} in the end-to-end loop: {tcg.last_error()}")
    return {"value": case.flops / (ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": n,
            "path": "pinned host A, B, C, bias, block scales -> device (cudaMemcpyAsync), " +
                    ("tcg_gemm_grouped" if is_grouped(case) else "tcg_gemm") + ", D -> pinned host; "
                    "steps pipelined over two device buffer sets (copies of step i+1 overlap the GEMM of step i)"}


def run_role_stats(args):
    """The kernel's cycle accounting (KernelParams::stats): summed over the CTAs
    of --steps launches, reported per issuing CTA and launch in microseconds at
    the SM clock sampled meanwhile.  The accounting slows the kernel a little,
    so these runs give no bench value."""
    os.environ["TCG_STATS"] = "1"           # read once, when the library loads
    import torch
    import tiled_tensor_core_persistent_gb300 as tcg
    from tiled_tensor_core_persistent_gb300 import _build, harness, inputs
    _build.build()
    tcg.lib()
    case = WORKLOADS[args.workload][0](inputs)
    dc = (harness.GroupedDeviceCase if is_grouped(case) else harness.DeviceCase)(case, device="cuda:0")
    for _ in range(max(args.warmup, 3)):
        dc.run()
    torch.cuda.synchronize()
    dc.workspace[:256].zero_()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        dc.run()
    ev1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    st = dc.workspace[64:128].view(torch.int64).cpu().tolist()
    mhz = clocks.get("sm_mhz") or 1900.0
    if is_grouped(case):
        plan = tcg.grouped_plan([dict(M=p.M, N=p.N, K=p.K) for p in case.problems], head(case).ab_dtype)
    else:
        plan = tcg.plan(case.M, case.N, case.K, dc.ab_dtype, case.opA, case.opB)
    issuers = max(st[6], 1)                 # MMA-issuing CTAs (pair leaders) summed over the launches
    ctas = issuers * plan["cluster"]        # every CTA: producers and epilogues count in each
    per = {"mma_wait_full": (st[0], issuers), "mma_wait_acc": (st[1], issuers), "mma_loop_total": (st[5], issuers),
           "producer_wait_empty": (st[2], ctas), "epilogue_wait_acc": (st[3], ctas), "epilogue_busy": (st[4], ctas)}
    print(json.dumps({"workload": args.workload, "launches": args.steps,
                      "ms_per_launch": ev0.elapsed_time(ev1) / args.steps, "sm_mhz": mhz, "plan": plan,
                      "us_per_cta_and_launch": {k: c / n / mhz for k, (c, n) in per.items()},
                      "note": "mma_* from the MMA issuer (first wait to last commit for mma_loop_total), "
                              "producer_* from the TMA producer, epilogue_* from the first epilogue warp of each "
                              "CTA (busy = accumulator ready to hand-back)"}), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.role_stats:
        return run_role_stats(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
