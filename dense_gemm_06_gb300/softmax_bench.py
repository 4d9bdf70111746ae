"""Row-softmax bandwidth on the Gluon Multi-CTA tutorial's benchmark shapes.

    python -m dense_gemm_06_gb300.softmax_bench [--reps 20] [--no-graph] [--shape M N]

For each shape (M rows of N fp32 values) prints the CTAs per row, the time per
call and the bandwidth counted as the tutorial counts it: 2 * M * N * 4 bytes
(one read of x, one write of y) per call. Like the tutorial's benchmark, the
time is taken over a CUDA graph of 10 back-to-back calls (CUDA events around
each replay, median of `reps` replays, after warm-up); --no-graph times
single calls instead. Inputs are seeded U[-1, 1) values.
"""

from __future__ import annotations

import argparse
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SHAPES = [(2 ** 15, 2 ** 8), (2 ** 15, 2 ** 9), (2 ** 15, 2 ** 10), (2 ** 15, 2 ** 11),
          (2 ** 15, 2 ** 12), (2 ** 15, 2 ** 13), (2 ** 15, 2 ** 14), (2 ** 15, 2 ** 15),
          (2 ** 15, 2 ** 16), (2 ** 14, 2 ** 17), (2 ** 13, 2 ** 18)]


GRAPH_CALLS = 10


def ctas_per_row(N: int) -> int:
    """CTAs per row as softmax_rows lays out 16-byte-aligned rows: one CTA up
    to 16384 columns, then a cluster of 16384-column CTAs."""
    cs = 1
    while cs * 16384 < N:
        cs *= 2
    return cs


def main(argv=None):
    import torch

    import datagen
    import dense_gemm_06_gb300 as lg

    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time single calls instead of a CUDA graph of back-to-back calls")
    ap.add_argument("--shape", type=int, nargs=2, metavar=("M", "N"),
                    help="run this one shape instead of the tutorial's list")
    a = ap.parse_args(argv)
    lg.load()
    torch.cuda.set_device(0)
    s = torch.cuda.Stream()
    print("   shape           CTAs/row  time (ms)  bandwidth (GB/s)")
    for M, N in ([tuple(a.shape)] if a.shape else SHAPES):
        x = torch.from_numpy(datagen.logical(M, N, dtype="f32", dist="pm1", seed=M ^ N)).cuda()
        y = torch.empty_like(x)
        cs = ctas_per_row(N)
        for _ in range(3):
            lg.check(lg.softmax_rows(M, N, x, N, y, N, s.cuda_stream))
        s.synchronize()
        times = []
        if a.graph:
            # the tutorial's method: back-to-back calls replayed from a CUDA
            # graph, so host launch gaps do not count
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(GRAPH_CALLS):
                    lg.check(lg.softmax_rows(M, N, x, N, y, N, s.cuda_stream))
            with torch.cuda.stream(s):  # replay() launches on the current stream
                g.replay()
                s.synchronize()
                for _ in range(a.reps):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(s)
                    g.replay()
                    e1.record(s)
                    s.synchronize()
                    times.append(e0.elapsed_time(e1) / GRAPH_CALLS)
            del g
        else:
            for _ in range(a.reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                lg.check(lg.softmax_rows(M, N, x, N, y, N, s.cuda_stream))
                e1.record(s)
                s.synchronize()
                times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        print(f"{M:>7} x {N:<7} {cs:>6}  {ms:>9.3f}  {2 * M * N * 4 / (ms * 1e-3) / 1e9:>16.1f}")
        del x, y


if __name__ == "__main__":
    main()
