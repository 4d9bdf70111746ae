"""Run one GEMM workload a few times through the C ABI, for profilers.

    python -m dense_gemm_06_gb300.profile_case --case sgemm --n 8192 --am 0 --bm 0 --reps 3
    python -m dense_gemm_06_gb300.profile_case --case bf16 --n 8192 --reps 3
    python -m dense_gemm_06_gb300.profile_case --case f16skinny --reps 3
    python -m dense_gemm_06_gb300.profile_case --case f16small --reps 3
    python -m dense_gemm_06_gb300.profile_case --case every
    python -m dense_gemm_06_gb300.profile_case --case bf16 --vendor --reps 2
    python -m dense_gemm_06_gb300.profile_case --case f16skinny --dtype 3 --bm 0 --vendor --reps 2

--case every runs one small call of each kernel of the library (for a
launch list that covers all of them): the tcgen05 GEMM at its small and
ragged shapes (with the operand repack), the TMA-fed FFMA kernel with its
K-slice tail and fixup, its stream-K variant, the cp.async FFMA kernel, the
transpose pre-pass, the K = 0 kernels of gemm, gemm_ex and gemm_noalloc,
gemm_noalloc's repack and the three row-softmax kernels.

Inputs are the seeded synthetic operands of the benchmark (datagen), resident
on the device before the first launch; each repetition is one gemm() call on
one stream, so a profiler sees exactly `reps` launches of the kernel (plus a
repack launch per misaligned operand for the ragged case). Prints the
CUDA-event time of every repetition (not a benchmark number).

--vendor runs torch.matmul (cuBLAS) on the same device operands instead of
the library, for a side-by-side capture of the vendor kernel (16-bit inputs
and C, both operands K-major). It is a comparison point for profiles,
never a path of the library.
"""

from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

CASES = {
    # name: (M, N, K, dtype, a_major, b_major, dist, seed, lo, hi)
    "sgemm": (8192, 8192, 8192, 0, 0, 0, "normal", 1027, 0, 0),
    "bf16": (8192, 8192, 8192, 4, 0, 0, "normal", 1028, 0, 0),
    "f16small": (1024, 512, 256, 1, 0, 0, "int", 1025, -5, 5),
    "sgemm2048": (2048, 2048, 2048, 0, 1, 1, "pm1", 1026, 0, 0),
    "f16ragged": (4095, 3071, 1037, 1, 0, 1, "int", 1029, -3, 3),
    "f16skinny": (16384, 256, 8192, 1, 0, 1, "int", 1030, -3, 3),
    # 20 x 16 = 320 tiles of 128 x 128: a 16-tile last wave on 304 FFMA CTA slots
    "sgemmtail": (2560, 2048, 8192, 0, 1, 1, "normal", 1031, 0, 0),
}


def run_every():
    """One small call of every kernel of the library (see the module doc)."""
    import torch

    import datagen
    import dense_gemm_06_gb300 as lg

    torch.cuda.set_device(0)
    lg.load()

    def dev(M, K, major, it, dist, seed, stream, pad=0, lo=-3, hi=3):
        ld = (K if major == 0 else M) + pad
        a = datagen.operand(M, K, major=major, ld=ld, dtype=it, dist=dist, seed=seed,
                            stream=stream, lo=lo, hi=hi)
        return torch.from_numpy(a.view(np.int16) if it != "f32" else a).cuda(), ld

    def run(what, M, N, K, dtype, am, bm, pad=0, opts=(), fn=None, ldc=None):
        it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
        dA, lda = dev(M, K, am, it, "int", 7, 0, pad)
        dB, ldb = dev(N, K, bm, it, "int", 7, 1, pad)
        ldc = ldc or N
        dC = torch.zeros(M * ldc, dtype=torch.float32 if ot == "f32" else torch.int16,
                         device="cuda")
        saved = [(o, lg.gemm_get_option(o)) for o, _ in opts]
        for o, v in opts:
            lg.check(lg.gemm_set_option(o, v))
        try:
            lg.check((fn or lg.gemm)(M, N, K, dA, lda, am, dB, ldb, bm, dC, ldc, 1, dtype), what)
            lg.check(lg.gemm_check_device_error(), what)
        finally:
            for o, v in saved:
                lg.gemm_set_option(o, v)
        print(f"every: {what}", flush=True)

    run("tcgen05, 1024x512x256 bf16 (one CTA per 128x64 tile)", 1024, 512, 256,
        lg.GEMM_BF16_F32, 0, 0)
    run("tcgen05 + repack, 1000x777x1037 fp16, misaligned A, B, C", 1000, 777, 1037,
        lg.GEMM_F16_F32, 0, 1, pad=1, ldc=779)
    run("FFMA TMA-fed + K-slice fixup, 1024x1024x8192", 1024, 1024, 8192, lg.GEMM_F32, 1, 1)
    run("FFMA TMA-fed stream-K, 2048^3", 2048, 2048, 2048, lg.GEMM_F32, 1, 1)
    run("FFMA cp.async (configuration 7), 300x520x200 K-major", 300, 520, 200, lg.GEMM_F32, 0,
        0, opts=((lg.GEMM_OPT_SIMT_CONFIG, 7),))
    run("transpose pre-pass + FFMA, 1024^3 K-major", 1024, 1024, 1024, lg.GEMM_F32, 0, 0,
        opts=((lg.GEMM_OPT_SIMT_TRANSPOSE, 2),))
    run("K = 0 (zero fill)", 300, 500, 0, lg.GEMM_F32, 0, 0)
    run("gemm_noalloc + its repack, 1000x777x1037 fp16 misaligned", 1000, 777, 1037,
        lg.GEMM_F16_F32, 0, 1, pad=1, fn=lg.gemm_noalloc)
    run("gemm_noalloc K = 0", 300, 500, 0, lg.GEMM_F16_F32, 0, 0, fn=lg.gemm_noalloc)
    C = torch.ones(300 * 500, dtype=torch.float32, device="cuda")
    lg.check(lg.gemm_ex(300, 500, 0, 0, 1, 0, 0, 1, 0, C, 500, 1, lg.GEMM_F32, beta=0.5),
             "gemm_ex K = 0")
    print("every: gemm_ex K = 0 (epilogue only)", flush=True)
    for M, N in ((4096, 512), (4096, 8192), (256, 65536), (256, 65537)):
        x = torch.randn(M * N, dtype=torch.float32, device="cuda")
        y = torch.empty_like(x)
        lg.check(lg.softmax_rows(M, N, x, N, y, N), "softmax_rows")
        print(f"every: softmax_rows {M} x {N}", flush=True)
    lg.check(lg.gemm_check_device_error(), "device error word")


def main(argv=None):
    import torch

    import datagen
    import dense_gemm_06_gb300 as lg

    if argv is None:
        argv = sys.argv[1:]
    if "--case" in argv and argv[argv.index("--case") + 1:argv.index("--case") + 2] == ["every"]:
        run_every()
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=sorted(CASES) + ["every"], required=True)
    ap.add_argument("--n", type=int, default=None, help="override M = N = K")
    ap.add_argument("--shape", type=int, nargs=3, metavar=("M", "N", "K"), default=None,
                    help="override M, N and K")
    ap.add_argument("--dtype", type=int, default=None, help="override the GEMM_* data type")
    ap.add_argument("--am", type=int, default=None)
    ap.add_argument("--bm", type=int, default=None)
    ap.add_argument("--cta-group", type=int, default=0)
    ap.add_argument("--simt-config", type=int, default=0)
    ap.add_argument("--tc-store", type=int, default=0)
    ap.add_argument("--tc-scheduler", type=int, default=0,
                    help="1 static persistent, 2 cluster launch control (0: automatic)")
    ap.add_argument("--simt-split", type=int, default=0,
                    help="FFMA last-wave K-split: 1 never, 2 always (0: automatic)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--vendor", action="store_true",
                    help="run torch.matmul (cuBLAS) on the same operands instead")
    ap.add_argument("--tune", action="store_true",
                    help="run gemm_tune first (records the fastest configuration)")
    a = ap.parse_args(argv)
    M, N, K, dtype, am, bm, dist, seed, lo, hi = CASES[a.case]
    if a.n:
        M = N = K = a.n
    if a.shape:
        M, N, K = a.shape
    dtype = dtype if a.dtype is None else a.dtype
    am = am if a.am is None else a.am
    bm = bm if a.bm is None else a.bm
    it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
    lda = K if am == 0 else M
    ldb = K if bm == 0 else N
    A = datagen.operand(M, K, major=am, ld=lda, dtype=it, dist=dist, seed=seed, stream=0,
                        lo=lo, hi=hi)
    B = datagen.operand(N, K, major=bm, ld=ldb, dtype=it, dist=dist, seed=seed, stream=1,
                        lo=lo, hi=hi)
    torch.cuda.set_device(0)
    lg.load()
    conv = (lambda x: x.view(np.int16)) if it != "f32" else (lambda x: x)
    dA = torch.from_numpy(conv(A)).cuda()
    dB = torch.from_numpy(conv(B)).cuda()
    dC = torch.empty(M * N, dtype=torch.float32 if ot == "f32" else torch.int16, device="cuda")
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_CTA_GROUP, a.cta_group))
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, a.simt_config))
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_STORE, a.tc_store))
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_SCHEDULER, a.tc_scheduler))
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, a.simt_split))
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    if a.tune:
        rc, t = lg.gemm_tune(M, N, K, dA, lda, am, dB, ldb, bm, dC, N, 1, dtype, 5,
                             s.cuda_stream)
        lg.check(rc, "gemm_tune")
        print(f"{a.case} {M}x{N}x{K} A{'KM'[am]} B{'KN'[bm]} tuned: {t}")
    if a.vendor:
        if it == "f32" or ot == "f32" or am != 0 or bm != 0:
            raise SystemExit("--vendor: 16-bit inputs and C, both operands K-major")
        tt = torch.bfloat16 if it == "bf16" else torch.float16
        tA, tB = dA.view(tt).view(M, K), dB.view(tt).view(N, K)
        tC = dC.view(tt).view(M, N)
    for r in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        if a.vendor:
            with torch.cuda.stream(s):
                torch.matmul(tA, tB.t(), out=tC)
        else:
            lg.check(lg.gemm(M, N, K, dA, lda, am, dB, ldb, bm, dC, N, 1, dtype,
                             s.cuda_stream))
        e1.record(s)
        s.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"{a.case} {M}x{N}x{K} rep {r}: {ms:.3f} ms, "
              f"{2.0 * M * N * K / (ms * 1e-3) / 1e12:.1f} TFLOP/s")
    lg.check(lg.gemm_check_device_error(s.cuda_stream))


if __name__ == "__main__":
    main()
