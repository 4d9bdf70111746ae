"""Every GEMM workload of the benchmark definition, timed per call.

    python -m dense_gemm_06_gb300.config_table [--warmup 10] [--reps 50]

Workloads: fp16 integers 1024x512x256 (A, B K-major, fp32 C); fp32 2048^3
(A M-major, B N-major); fp32 8192^3 in all four A/B majors; bf16 8192^3
(bf16 C); fp16 integers 4095x3071x1037 (A K-major, B N-major, packed) and
16384x256x8192. Each is timed with CUDA events around single gemm() calls on
one stream: `warmup` untimed calls, then `reps` timed ones, reporting the
median and the minimum. Hot: the same operands every call. Cold: as many
device copies of A, B and C as make the set exceed twice the L2 size, used in
turn (a workload whose operands already exceed that runs hot only). TFLOP/s
= 2 M N K / t; the roof of each workload is the FP32-FFMA peak (SMs x 128
lanes x 2 x max SM clock) for fp32, the dense 16-bit tensor peak for 16-bit,
or, where the arithmetic intensity (flop per compulsory byte) times the
measured HBM bandwidth is lower, that. The SM clock is sampled before and
after. Prints a markdown table and one JSON line per workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# (name, M, N, K, dtype, a_major, b_major, distribution, seed, lo, hi)
WORKLOADS = [
    ("fp16 int 1024x512x256, A K B K, C fp32", 1024, 512, 256, 1, 0, 0, "int", 1025, -5, 5),
    ("fp32 2048^3, A M B N", 2048, 2048, 2048, 0, 1, 1, "pm1", 1026, 0, 0),
    ("fp32 8192^3, A K B K", 8192, 8192, 8192, 0, 0, 0, "normal", 1027, 0, 0),
    ("fp32 8192^3, A K B N", 8192, 8192, 8192, 0, 0, 1, "normal", 1027, 0, 0),
    ("fp32 8192^3, A M B K", 8192, 8192, 8192, 0, 1, 0, "normal", 1027, 0, 0),
    ("fp32 8192^3, A M B N", 8192, 8192, 8192, 0, 1, 1, "normal", 1027, 0, 0),
    ("bf16 8192^3, A K B K, C bf16", 8192, 8192, 8192, 4, 0, 0, "normal", 1028, 0, 0),
    ("fp16 int 4095x3071x1037, A K B N, C fp32", 4095, 3071, 1037, 1, 0, 1, "int", 1029, -3, 3),
    ("fp16 int 16384x256x8192, A K B N, C fp32", 16384, 256, 8192, 1, 0, 1, "int", 1030, -3, 3),
]


def sm_clock_mhz():
    """(current, max) SM clock of GPU 0 from nvidia-smi, or (None, None)."""
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm",
                              "--format=csv,noheader,nounits", "-i", "0"],
                             capture_output=True, text=True, timeout=20).stdout
        cur, mx = (float(v) for v in out.strip().split(","))
        return cur, mx
    except Exception:
        return None, None


def measured_peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, source) from MEASURED_PEAKS.json,
    else the fallback figures."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def time_calls(call, warmup, reps, stream, torch):
    """Median and minimum (ms) of `reps` single calls after `warmup` ones;
    call(i) issues the i-th call on `stream`."""
    for i in range(warmup):
        call(i)
    stream.synchronize()
    times = []
    for i in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call(warmup + i)
        e1.record(stream)
        stream.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times), min(times)


def main(argv=None):
    import numpy as np
    import torch

    import datagen
    import dense_gemm_06_gb300 as lg

    ap = argparse.ArgumentParser()
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--reps", type=int, default=50)
    a = ap.parse_args(argv)
    lg.load()
    torch.cuda.set_device(0)
    prop = torch.cuda.get_device_properties(0)
    l2 = int(getattr(prop, "L2_cache_size", 0) or 129 * 2 ** 20)
    clk0, clk_max = sm_clock_mhz()
    f_ghz = (clk_max or 2070.0) / 1e3
    ffma_peak = prop.multi_processor_count * 128 * 2 * f_ghz / 1e3  # TFLOP/s
    hbm, tc_peak, src = measured_peaks()
    s = torch.cuda.Stream()
    rows = []
    for name, M, N, K, dtype, am, bm, dist, seed, lo, hi in WORKLOADS:
        it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
        ie, oe = (4 if it == "f32" else 2), (4 if ot == "f32" else 2)
        lda, ldb = (K if am == 0 else M), (K if bm == 0 else N)
        A = datagen.operand(M, K, major=am, ld=lda, dtype=it, dist=dist, seed=seed, stream=0,
                            lo=lo, hi=hi)
        B = datagen.operand(N, K, major=bm, ld=ldb, dtype=it, dist=dist, seed=seed, stream=1,
                            lo=lo, hi=hi)
        set_bytes = A.size * ie + B.size * ie + M * N * oe
        copies = 1 if set_bytes > 2 * l2 else -(-2 * l2 // set_bytes) + 1
        conv = (lambda x: torch.from_numpy(x.view(np.int16))) if ie == 2 else torch.from_numpy
        dA = [conv(A).cuda() for _ in range(copies)]
        dB = [conv(B).cuda() for _ in range(copies)]
        cdt = torch.float32 if oe == 4 else torch.int16
        dC = [torch.empty(M * N, dtype=cdt, device="cuda") for _ in range(copies)]

        def call(i, j=None):
            k = (i % copies) if j is None else j
            lg.check(lg.gemm(M, N, K, dA[k], lda, am, dB[k], ldb, bm, dC[k], N, 1, dtype,
                             s.cuda_stream), name)

        hot = time_calls(lambda i: call(i, 0), a.warmup, a.reps, s, torch)
        cold = time_calls(call, a.warmup, a.reps, s, torch) if copies > 1 else None
        lg.check(lg.gemm_check_device_error(s.cuda_stream), name)
        flops = 2.0 * M * N * K
        ai = flops / set_bytes
        if dtype == 0:
            roof, kind = ffma_peak, "FFMA"
        elif ai * hbm / 1e3 < tc_peak:
            roof, kind = ai * hbm / 1e3, "HBM (AI x BW)"
        else:
            roof, kind = tc_peak, "tensor"
        tf = flops / (hot[0] * 1e-3) / 1e12
        row = {"workload": name, "median_ms": round(hot[0], 4), "min_ms": round(hot[1], 4),
               "tflops_median": round(tf, 2), "roof_tflops": round(roof, 1), "roof": kind,
               "frac_of_roof": round(tf / roof, 4), "arith_intensity": round(ai, 1),
               "cold_l2": None if cold is None else {
                   "copies": copies, "median_ms": round(cold[0], 4), "min_ms": round(cold[1], 4),
                   "tflops_median": round(flops / (cold[0] * 1e-3) / 1e12, 2)}}
        rows.append(row)
        del dA, dB, dC
        torch.cuda.empty_cache()
    clk1, _ = sm_clock_mhz()
    print(f"SM clock before/after: {clk0} / {clk1} MHz (max {clk_max}); FFMA peak "
          f"{ffma_peak:.2f} TFLOP/s (derived), tensor peak {tc_peak} TFLOP/s and HBM {hbm} GB/s "
          f"({src}); {a.warmup} warm-up + {a.reps} timed calls each")
    print("| workload | median ms | min ms | TFLOP/s | roof | % of roof | cold-L2 median ms |")
    print("|---|---|---|---|---|---|---|")
    for r in rows:
        cold = r["cold_l2"]["median_ms"] if r["cold_l2"] else "(operands > 2 x L2)"
        print(f"| {r['workload']} | {r['median_ms']} | {r['min_ms']} | {r['tflops_median']} | "
              f"{r['roof']} {r['roof_tflops']} | {100 * r['frac_of_roof']:.1f}% | {cold} |")
    for r in rows:
        print(json.dumps(r))


if __name__ == "__main__":
    main()
