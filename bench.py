"""Benchmark: GEMM TFLOP/s at 8192^3 on one GB300.

One step is one pass of the whole hot path over one batch of seeded
synthetic inputs: the 8192^3 fp32 SGEMM on the FFMA kernel for each of the
four A/B major combinations (C N-major), then the 8192^3 bf16 -> bf16 GEMM
(A, B K-major) on the tcgen05 kernel -- the fp32 workload of the CuTe DSL
Ampere SGEMM example's ncu recipe and the 8192 x 8192 x 8192 point of the
Gluon Multi-CTA tutorial's matmul benchmark.

    value        = 5 * 2 * 8192^3 * steps / (device time of the timed steps),
                   inputs resident in HBM
    e2e          = the same through gemm_host(): pinned host A, B in, host C
                   out, copies inside the timed region
    roofline     = the dominant kernel (the FFMA SGEMM) against its ALU peak
    cpu_baseline = the fp64 CPU oracle on a bounded sample of the workload

Usage: python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl native|reference]
The library runs on one GPU (its opt-in cluster-multicast TMA variant must
only ever address this GPU's memory), so --gpus accepts 1 only.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s and % of FP32-FFMA / BF16-tensor peak at 8192³, 1×GB300"
UNIT = "TFLOP/s"
NDIM = 8192
SEED_F32, SEED_BF16 = 1027, 1028
FLOPS_PER_GEMM = 2.0 * NDIM ** 3
WORKLOAD = ("8192^3 fp32 SGEMM x 4 A/B majors (C N-major, FFMA kernel) + 8192^3 bf16->bf16 "
            "GEMM (A,B K-major, tcgen05 2-CTA kernel); one step = these 5 GEMMs")

# Peaks. FFMA: SMs x 128 fp32 lanes x 2 flop x maximum SM clock, from the SM
# count the device reports and the maximum clock nvidia-smi reports during the
# run; GB300's 152 SMs and 2.07 GHz when either is unavailable.
SMS, FP32_LANES, SM_MAX_GHZ = 152, 128, 2.07
FFMA_PEAK_TFLOPS = SMS * FP32_LANES * 2 * SM_MAX_GHZ / 1e3
SGEMM_KERNEL = "sgemm_ffma_tma_kernel"  # the FFMA kernel the step's fp32 GEMMs run


def ffma_peak(sm_count, sm_max_mhz):
    """(TFLOP/s, how it was obtained) of the FP32 FFMA pipe."""
    sms = int(sm_count) if sm_count else SMS
    ghz = float(sm_max_mhz) / 1e3 if sm_max_mhz else SM_MAX_GHZ
    how = (f"derived: {sms} SMs ({'queried' if sm_count else 'assumed'}) x {FP32_LANES} FP32 "
           f"lanes x 2 x {ghz:.3g} GHz ({'nvidia-smi max SM clock' if sm_max_mhz else 'assumed'})")
    return sms * FP32_LANES * 2 * ghz / 1e3, how
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------- inputs --

def make_inputs():
    """Host storage of the step's operands (seeded; see datagen)."""
    import datagen
    LA = datagen.logical(NDIM, NDIM, dtype="f32", dist="normal", seed=SEED_F32, stream=0)
    LB = datagen.logical(NDIM, NDIM, dtype="f32", dist="normal", seed=SEED_F32, stream=1)
    f32 = {"A0": LA, "A1": np.ascontiguousarray(LA.T), "B0": LB, "B1": np.ascontiguousarray(LB.T)}
    bf = {"A": datagen.logical(NDIM, NDIM, dtype="bf16", dist="normal", seed=SEED_BF16, stream=0),
          "B": datagen.logical(NDIM, NDIM, dtype="bf16", dist="normal", seed=SEED_BF16, stream=1)}
    return f32, bf


GEMMS = [("fp32 A K-major B K-major", 0, 0), ("fp32 A K-major B N-major", 0, 1),
         ("fp32 A M-major B K-major", 1, 0), ("fp32 A M-major B N-major", 1, 1)]


# ------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(dev_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(dev_index)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.remove(self.path)
        return summarize_clocks(lines)


CLOCK_REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def summarize_clocks(lines):
    """Median SM clock under load, max clock and the throttle reasons seen,
    from nvidia-smi CSV rows (ClockSampler.FIELDS, no header, no units)."""
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 7:
            continue
        try:
            rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
        except ValueError:
            continue
    if not rows:
        return None
    sm = [r[0] for r in rows]
    reasons = sorted({CLOCK_REASONS[i] for r in rows for i, v in enumerate(r[2])
                      if v == "Active"})
    loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
            "reasons": reasons, "samples": len(rows)}


def throughput_tflops(flops_per_step, steps, ms):
    """TFLOP/s of `steps` steps of `flops_per_step` that took `ms` of device time."""
    return flops_per_step * steps / (ms * 1e-3) / 1e12


# ------------------------------------------------------- native arm --

def run_native(args):
    import torch

    import dense_gemm_06_gb300 as lg

    torch.cuda.set_device(0)
    lg.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    s_handle = stream.cuda_stream

    f32, bf = make_inputs()
    d = {k: torch.from_numpy(v).to(dev) for k, v in f32.items()}
    dA16 = torch.from_numpy(bf["A"].view(np.int16)).to(dev)
    dB16 = torch.from_numpy(bf["B"].view(np.int16)).to(dev)
    C32 = torch.empty(NDIM * NDIM, dtype=torch.float32, device=dev)
    C16 = torch.empty(NDIM * NDIM, dtype=torch.int16, device=dev)
    torch.cuda.synchronize()

    n = NDIM
    n_gemms = len(GEMMS) + 1
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_gemms + 1)]
          for _ in range(args.steps)]

    def step(events=None):
        if events:
            events[0].record(stream)
        for i, (_, am, bm) in enumerate(GEMMS):
            lg.check(lg.gemm(n, n, n, d[f"A{am}"], n, am, d[f"B{bm}"], n, bm, C32, n, 1,
                             lg.GEMM_F32, s_handle))
            if events:
                events[i + 1].record(stream)
        lg.check(lg.gemm(n, n, n, dA16, n, 0, dB16, n, 0, C16, n, 1, lg.GEMM_BF16_BF16,
                         s_handle))
        if events:
            events[n_gemms].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    lg.check(lg.gemm_check_device_error(s_handle), "device error word")

    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    launches0 = lg.gemm_launch_count()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            step(ev[k])
    t_end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    launches = lg.gemm_launch_count() - launches0
    lg.check(lg.gemm_check_device_error(s_handle), "device error word")

    ms_total = t_start.elapsed_time(t_end)
    per = np.array([[ev[k][i].elapsed_time(ev[k][i + 1]) for i in range(n_gemms)]
                    for k in range(args.steps)])
    per_ms = per.mean(axis=0)

    parity = sampled_parity(C16, C32, f32, bf, d, lg, s_handle)

    # e2e through the host-buffer entry point (pinned host memory)
    e2e = run_e2e(args, lg, f32, bf, stream)

    peaks, peak_src = load_peaks()
    ffma_tf, ffma_how = ffma_peak(torch.cuda.get_device_properties(dev).multi_processor_count,
                                  (clocks or {}).get("sm_max_mhz"))
    flops_step = FLOPS_PER_GEMM * n_gemms
    value = throughput_tflops(flops_step, args.steps, ms_total)
    parts = []
    for i, (name, am, bm) in enumerate(GEMMS):
        tf = FLOPS_PER_GEMM / (per_ms[i] * 1e-3) / 1e12
        parts.append({"gemm": name, "kernel": SGEMM_KERNEL, "ms": round(per_ms[i], 4),
                      "tflops": round(tf, 2), "peak_tflops": round(ffma_tf, 2),
                      "peak_kind": "alu (FFMA, derived)", "frac": round(tf / ffma_tf, 4)})
    tf16 = FLOPS_PER_GEMM / (per_ms[-1] * 1e-3) / 1e12
    parts.append({"gemm": "bf16->bf16 A K-major B K-major", "kernel": "gemm_tc_kernel",
                  "ms": round(per_ms[-1], 4), "tflops": round(tf16, 2),
                  "peak_tflops": peaks["bf16_tflops"], "peak_kind": f"bf16 burst ({peak_src})",
                  "frac": round(tf16 / peaks["bf16_tflops"], 4),
                  "frac_of_sustained": round(tf16 / peaks["bf16_tflops_sustained"], 4)})
    # The kernel's own launch duration: the call with both operands MN-major
    # is one launch of the FFMA kernel and nothing else (the K-major calls
    # add the transpose pre-pass, which runs the same kernel afterwards).
    mn = next(i for i, (_, am, bm) in enumerate(GEMMS) if am == 1 and bm == 1)
    sgemm_ms = float(per_ms[mn])
    achieved = FLOPS_PER_GEMM / (sgemm_ms * 1e-3) / 1e12
    roofline = {"bound": "alu", "achieved": round(achieved, 2), "peak": round(ffma_tf, 2),
                "unit": "TFLOP/s", "frac": round(achieved / ffma_tf, 4),
                "traffic": profiled_traffic(SGEMM_KERNEL),
                "kernel": SGEMM_KERNEL,
                "timed_launches": f"{GEMMS[mn][0]} call of each timed step (one launch of "
                                  "the kernel per call, CUDA events on its stream)",
                "peak_source": ffma_how}
    roofline_tc = {"bound": "tensor", "achieved": round(tf16, 2), "peak": peaks["bf16_tflops"],
                   "unit": "TFLOP/s", "frac": round(tf16 / peaks["bf16_tflops"], 4),
                   "traffic": profiled_traffic("gemm_tc_kernel"), "kernel": "gemm_tc_kernel",
                   "peak_source": f"MEASURED_PEAKS bf16_tflops burst ({peak_src})"}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32+bf16",
        "data": "synthetic: seeded SplitMix64 N(0,1), fp32 (seed 1027) and bf16 (seed 1028)",
        "config": {"workload": WORKLOAD, "M": NDIM, "N": NDIM, "K": NDIM,
                   "gemms_per_step": n_gemms,
                   "l2": "no flush; every operand (256 MiB fp32, 128 MiB bf16) exceeds the "
                         "129 MB L2 and a step streams >2 GB",
                   "parallelism": "single GPU"},
        "roofline": roofline, "roofline_tc": roofline_tc, "parts": parts,
        "e2e": e2e, "gpu_launches": int(launches), "clocks": clocks, "parity": parity,
        "cpu_baseline": cpu_baseline(f32, bf) if not args.no_cpu_baseline else None,
    }
    print(json.dumps(line), flush=True)


def run_e2e(args, lg, f32, bf, stream):
    """The step through gemm_host(): pinned host operands in, host C out."""
    import torch
    n = NDIM
    h = {k: torch.from_numpy(v).pin_memory() for k, v in f32.items()}
    hA16 = torch.from_numpy(bf["A"].view(np.int16)).pin_memory()
    hB16 = torch.from_numpy(bf["B"].view(np.int16)).pin_memory()
    hC32 = torch.empty(n * n, dtype=torch.float32).pin_memory()
    hC16 = torch.empty(n * n, dtype=torch.int16).pin_memory()
    s = stream.cuda_stream

    def step():
        for _, am, bm in GEMMS:
            lg.check(lg.gemm_host(n, n, n, h[f"A{am}"], n, am, h[f"B{bm}"], n, bm, hC32, n, 1,
                                  lg.GEMM_F32, s), "gemm_host")
        lg.check(lg.gemm_host(n, n, n, hA16, n, 0, hB16, n, 0, hC16, n, 1, lg.GEMM_BF16_BF16, s),
                 "gemm_host")

    steps = max(1, min(args.steps, 5))
    for _ in range(max(1, min(args.warmup, 2))):
        step()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1)
    h2d = 4 * 2 * n * n * 4 + 2 * n * n * 2
    d2h = 4 * n * n * 4 + n * n * 2
    return {"value": round(throughput_tflops(FLOPS_PER_GEMM * 5, steps, ms), 3),
            "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": round(ms / steps, 3),
            "api": "gemm_host (C ABI, pinned host buffers)"}


def sampled_parity(C16, C32, f32, bf, d, lg, s_handle):
    """Checks 8 seeded rows of the last fp32 GEMM and of the bf16 GEMM
    against the oracle (the full parity suite lives in tests/)."""
    import torch

    import datagen
    import oracle
    from tests.acceptance import violations
    n = NDIM
    rows = datagen.sample_indices(n, 6, seed=77)
    torch.cuda.synchronize()
    out = {}
    c32 = C32.view(n, n)[torch.from_numpy(rows).to(C32.device)].cpu().numpy().astype(np.float64)
    Cr, Sr = oracle.gemm_ref(n, n, n, f32["A1"].ravel(), n, 1, "f32", f32["B1"].ravel(), n, 1,
                             "f32", rows=rows)
    bad, worst = violations(c32, Cr, Sr, "f32")
    out["fp32_rows"] = {"rows": len(rows), "bad": int(bad.sum()), "worst_err_over_bound": worst}
    c16 = C16.view(n, n)[torch.from_numpy(rows).to(C16.device)].cpu().numpy()
    c16 = (c16.view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    Cr, Sr = oracle.gemm_ref(n, n, n, bf["A"].ravel(), n, 0, "bf16", bf["B"].ravel(), n, 0,
                             "bf16", rows=rows)
    bad, worst = violations(c16, Cr, Sr, "bf16")
    out["bf16_rows"] = {"rows": len(rows), "bad": int(bad.sum()), "worst_err_over_bound": worst}
    out["ok"] = out["fp32_rows"]["bad"] == 0 and out["bf16_rows"]["bad"] == 0
    return out


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)[kernel]
    except Exception:
        return None
    names = entry["source"] if isinstance(entry["source"], list) else [entry["source"]]
    h = hashlib.sha256()
    try:
        for name in names:  # the kernel's sources, hashed in the listed order
            with open(os.path.join(ROOT, "dense_gemm_06_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    digest = h.hexdigest()[:16]
    return entry["bytes_per_launch"] if digest == entry["source_sha256_16"] else None


# ------------------------------------------------------ CPU baselines --

CPU_ROWS = 400  # rows of each 8192^3 GEMM the oracle computes per sample (~10 s)
# Reference arm: rows per timed step (~5 s on 16 host cores, so 10 steps plus
# warm-up take about a minute; fewer rows would mostly time the decoding of B)
REF_ROWS = 256


def oracle_sample(f32, bf, rows_per_gemm, per_gemm=None):
    """The oracle on `rows_per_gemm` seeded rows of each of the step's GEMMs;
    returns (flops, seconds). per_gemm, if a list, receives (name, seconds)."""
    import datagen
    import oracle
    n = NDIM
    rows = datagen.sample_indices(n, rows_per_gemm, seed=55, always=())
    t0 = time.perf_counter()
    for name, am, bm in GEMMS:
        t = time.perf_counter()
        oracle.gemm_ref(n, n, n, f32[f"A{am}"].ravel(), n, am, "f32", f32[f"B{bm}"].ravel(), n,
                        bm, "f32", rows=rows)
        if per_gemm is not None:
            per_gemm.append((name, time.perf_counter() - t))
    t = time.perf_counter()
    oracle.gemm_ref(n, n, n, bf["A"].ravel(), n, 0, "bf16", bf["B"].ravel(), n, 0, "bf16",
                    rows=rows)
    if per_gemm is not None:
        per_gemm.append(("bf16->bf16 A K-major B K-major", time.perf_counter() - t))
    dt = time.perf_counter() - t0
    return 2.0 * len(rows) * n * n * (len(GEMMS) + 1), dt


# The smaller workloads of the benchmark definition, which the oracle runs in
# full for the per-workload baseline: (name, M, N, K, in type, a_major,
# b_major, distribution, seed, lo, hi).
SMALL_WORKLOADS = [
    ("fp16 int 1024x512x256, A K B K", 1024, 512, 256, "f16", 0, 0, "int", 1025, -5, 5),
    ("fp32 2048^3, A M B N", 2048, 2048, 2048, "f32", 1, 1, "pm1", 1026, 0, 0),
    ("fp16 int 4095x3071x1037, A K B N", 4095, 3071, 1037, "f16", 0, 1, "int", 1029, -3, 3),
    ("fp16 int 16384x256x8192, A K B N", 16384, 256, 8192, "f16", 0, 1, "int", 1030, -3, 3),
]


def oracle_small_workloads():
    """The oracle's fp64 rate on each small workload, computed in full."""
    import datagen
    import oracle
    out = []
    for name, M, N, K, it, am, bm, dist, seed, lo, hi in SMALL_WORKLOADS:
        lda, ldb = (K if am == 0 else M), (K if bm == 0 else N)
        A = datagen.operand(M, K, major=am, ld=lda, dtype=it, dist=dist, seed=seed, stream=0,
                            lo=lo, hi=hi)
        B = datagen.operand(N, K, major=bm, ld=ldb, dtype=it, dist=dist, seed=seed, stream=1,
                            lo=lo, hi=hi)
        t = time.perf_counter()
        oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, bm, it, with_s=False)
        dt = time.perf_counter() - t
        out.append({"workload": name, "seconds": round(dt, 3),
                    "gflops_fp64": round(2.0 * M * N * K / dt / 1e9, 2), "sample": "full"})
    return out


def cpu_baseline(f32, bf):
    """The oracle's rate on a bounded sample of every GEMM of the step, and
    each GEMM's full 8192^3 time extrapolated from it (2 M N K / rate)."""
    import oracle
    per = []
    flops, dt = oracle_sample(f32, bf, CPU_ROWS, per)
    one = 2.0 * CPU_ROWS * NDIM * NDIM
    full = 2.0 * NDIM ** 3
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{CPU_ROWS} seeded rows (all 8192 columns) of each of the step's 5 GEMMs "
                      f"({flops:.3g} flop, {dt:.1f} s), fp64 triple loop",
            "per_gemm": [{"gemm": name, "gflops_fp64": round(one / t / 1e9, 2),
                          "extrapolated_full_s": round(full / (one / t), 1)}
                         for name, t in per],
            "per_small_workload": oracle_small_workloads()}


def run_reference(args):
    """The reference arm: the CPU oracle timed on this machine's host cores on the
    same workload, each step a bounded sample of it."""
    import oracle
    f32, bf = make_inputs()
    rows = REF_ROWS
    for _ in range(args.warmup):
        oracle_sample(f32, bf, 2)
    tot_flops, tot_s = 0.0, 0.0
    for _ in range(args.steps):
        fl, dt = oracle_sample(f32, bf, rows)
        tot_flops += fl
        tot_s += dt
    value = tot_flops / tot_s / 1e12
    sample = (f"{rows} seeded rows (all 8192 columns) of each of the step's 5 GEMMs per step, "
              f"fp64 triple loop")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": NDIM, "N": NDIM, "K": NDIM,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1, choices=[1],
                    help="1 only: libgemm is a single-GPU library")
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "native":
        print("note: fewer than 3 warm-up steps do not meet the timing rules", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
