"""The library's per-(device, stream) scratch cache: the repack buffer of
misaligned 16-bit operands and the FFMA stream-K workspace are kept across
calls and reused by the next call on the same stream. Calls spread over more
streams than the cache holds (eviction), a call that needs a larger buffer
than its stream's (growth) and two host threads enqueueing on one stream
(the second finds the entry busy and takes a pool allocation) must all give
the oracle's result exactly: integer-valued inputs, fp32 accumulation."""

import threading

import numpy as np
import pytest

import dense_gemm_06_gb300 as lg
from gpu_util import CBuffer, check_full, make_operands, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


class Call:
    """One gemm() on given operands, C in a guarded buffer (A K-major, B
    N-major, C row-major; the pads make every pitch misaligned for TMA)."""

    def __init__(self, M, N, K, dtype, seed, pads=(1, 3, 1), am=0, bm=1):
        self.args = (M, N, K, dtype)
        self.am, self.bm = am, bm
        self.A, self.lda, self.B, self.ldb = make_operands(
            M, N, K, dtype, am, bm, "int", seed, lda_pad=pads[0], ldb_pad=pads[1], lo=-3, hi=3)
        self.dA, self.dB = to_device(self.A), to_device(self.B)
        self.ldc = N + pads[2]
        self.c = CBuffer(M, N, lg.GEMM_MAJOR_MN, self.ldc, lg.OUT_TYPE[dtype])

    def enqueue(self, stream):
        M, N, K, dtype = self.args
        rc = lg.gemm(M, N, K, self.dA, self.lda, self.am, self.dB, self.ldb, self.bm,
                     self.c.ptr(), self.ldc, lg.GEMM_MAJOR_MN, dtype, stream.cuda_stream)
        lg.check(rc, "gemm")

    def check(self, what):
        M, N, K, dtype = self.args
        check_full(self.c.read(), M, N, K, dtype, self.A, self.lda, self.am, self.B, self.ldb,
                   self.bm, exact=True, what=what)


def test_repack_buffers_across_more_streams_than_entries():
    import torch
    streams = [torch.cuda.Stream() for _ in range(11)]
    calls = [[Call(150 + 37 * i, 120 + 11 * i, 131 + 5 * i, lg.GEMM_F16_F32, seed=i),
              Call(90 + 7 * i, 300 + 3 * i, 77, lg.GEMM_BF16_F32, seed=100 + i)]
             for i in range(len(streams))]
    for rnd in range(2):  # the second round reuses (or re-creates) every stream's buffer
        for i, s in enumerate(streams):
            for c in calls[i]:
                c.enqueue(s)
        torch.cuda.synchronize()
        lg.check(lg.gemm_check_device_error(), "device error word")
        for i in range(len(streams)):
            for j, c in enumerate(calls[i]):
                c.check(f"round {rnd} stream {i} call {j}")


def test_repack_buffer_grows_on_its_stream():
    import torch
    s = torch.cuda.Stream()
    small = Call(64, 64, 33, lg.GEMM_F16_F32, seed=7)
    large = Call(1500, 1100, 517, lg.GEMM_F16_F32, seed=8)
    for c in (small, large, small):
        c.enqueue(s)
    torch.cuda.synchronize()
    small.check("small after large")
    large.check("large")


def test_two_threads_on_one_stream():
    import torch
    s = torch.cuda.Stream()
    calls = [[Call(300 + 29 * j, 211, 140 + 3 * j, lg.GEMM_F16_F32, seed=40 + 10 * t + j)
              for j in range(4)] for t in range(2)]
    errors = []

    def work(t):
        try:
            for c in calls[t]:
                c.enqueue(s)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    lg.check(lg.gemm_check_device_error(), "device error word")
    for t in range(2):
        for j, c in enumerate(calls[t]):
            c.check(f"thread {t} call {j}")


def test_stream_k_workspace_across_streams():
    import torch
    saved = lg.gemm_get_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL)
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 3))
    try:
        streams = [torch.cuda.Stream() for _ in range(3)]
        calls = [Call(1000 + 24 * i, 1024, 333, lg.GEMM_F32, seed=60 + i, pads=(0, 0, 0),
                      am=1, bm=1) for i in range(3)]
        for rnd in range(2):
            for c, s in zip(calls, streams):
                c.enqueue(s)
            torch.cuda.synchronize()
            lg.check(lg.gemm_check_device_error(), "device error word")
            for i, c in enumerate(calls):
                c.check(f"stream-K round {rnd} stream {i}")
    finally:
        lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, saved)


def test_graph_capture_takes_its_own_scratch():
    # A call captured into a CUDA graph must not bake in the stream's cached
    # buffer: replaying the graph and then running another misaligned call
    # eagerly on the same stream (which reuses the cached buffer) gives both
    # results exactly.
    import torch
    s = torch.cuda.Stream()
    a = Call(333, 277, 131, lg.GEMM_F16_F32, seed=90)
    b = Call(200, 150, 99, lg.GEMM_F16_F32, seed=91)
    a.enqueue(s)  # creates the stream's cache entry
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        a.enqueue(s)
    a.c.dev.copy_(torch.from_numpy(a.c.host_init.copy()).to(a.c.dev.device))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    b.enqueue(s)
    torch.cuda.synchronize()
    lg.check(lg.gemm_check_device_error(), "device error word")
    a.check("graph replay")
    b.check("eager call after the replay")
