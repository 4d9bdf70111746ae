"""gemm_noalloc(): the 16-bit GEMM for callers that cannot allocate device
memory (a program whose own allocator already holds the device memory, or a
loop where a device allocation is not acceptable). It repacks misaligned
operands into a fixed 32 MiB array inside the library instead of pool
scratch. These tests call it through the C ABI, several times in a row (the
array keeps the previous call's contents), and compare its C with the CPU
oracle under the acceptance rules: bit-exact for integer inputs, 1 ulp of
the output type + 1e-4 * sum|a*b| for float inputs.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test before it."""

import numpy as np
import pytest

import dense_gemm_06_gb300 as lg
import oracle
from acceptance import assert_accepted
from gpu_util import CBuffer, make_operands, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


def noalloc_vs_oracle(M, N, K, dtype, am, bm, cm, dist, seed, lda_pad, ldb_pad, ldc_pad,
                      lo=-5, hi=5):
    """Runs gemm_noalloc() on seeded inputs and checks C against the oracle."""
    import torch
    A, lda, B, ldb = make_operands(M, N, K, dtype, am, bm, dist, seed, lda_pad, ldb_pad, lo, hi)
    it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
    ldc = (N if cm == lg.GEMM_MAJOR_MN else M) + ldc_pad
    cbuf = CBuffer(M, N, cm, ldc, ot)
    lg.check(lg.gemm_noalloc(M, N, K, to_device(A), lda, am, to_device(B), ldb, bm, cbuf.ptr(),
                             ldc, cm, dtype), "gemm_noalloc")
    lg.check(lg.gemm_check_device_error(), "device error word")
    torch.cuda.synchronize()
    C = cbuf.read()
    C_ref, S = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, bm, it)
    assert_accepted(C, C_ref, S, ot, exact=(dist == "int"),
                    what=f"gemm_noalloc {M}x{N}x{K} dtype {dtype}")


def test_two_calls_in_a_row_match_the_oracle():
    # 1st call: both operands misaligned (lda 1037, ldb 777 elements), integer
    # fp16 -> fp32: the result is exact.
    noalloc_vs_oracle(1000, 777, 1037, lg.GEMM_F16_F32, 0, 1, 1, "int", 1029, 0, 0, 3,
                      lo=-3, hi=3)
    # 2nd call right after: another shape, type and layout, float data; the
    # array still holds the first call's operands.
    noalloc_vs_oracle(513, 1100, 333, lg.GEMM_BF16_BF16, 1, 0, 0, "normal", 31, 5, 3, 1)
    # 3rd call: the first problem again (the array now holds the second's data)
    noalloc_vs_oracle(1000, 777, 1037, lg.GEMM_F16_F32, 0, 1, 1, "int", 1029, 0, 0, 3,
                      lo=-3, hi=3)


def test_aligned_operands_and_k_zero():
    # aligned operands need no repack; K == 0 zero-fills C like gemm()
    noalloc_vs_oracle(300, 520, 128, lg.GEMM_F16_F16, 0, 0, 1, "int", 7, 0, 0, 0)
    import torch
    cbuf = CBuffer(37, 45, 1, 48, "f32")
    lg.check(lg.gemm_noalloc(37, 45, 0, 0, 1, 0, 0, 1, 0, cbuf.ptr(), 48, 1, lg.GEMM_BF16_F32),
             "gemm_noalloc")
    torch.cuda.synchronize()
    assert np.all(cbuf.read() == 0)


def test_rejects_problems_over_the_fixed_limit():
    import torch
    # A K-major 8192 x 2049 fp16 with lda 2049: repacked rows of 2056
    # elements take 8192 * 2056 * 2 bytes > 32 MiB
    M, N, K = 8192, 64, 2049
    dA = torch.zeros(M * K, dtype=torch.int16, device="cuda")
    dB = torch.zeros(N * K, dtype=torch.int16, device="cuda")
    dC = torch.zeros(M * N, dtype=torch.float32, device="cuda")
    n0 = lg.gemm_launch_count()
    rc = lg.gemm_noalloc(M, N, K, dA, K, 0, dB, K, 0, dC, N, 1, lg.GEMM_F16_F32)
    assert rc == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_launch_count() == n0
    assert lg.gemm_noalloc(4, 4, 4, dA, 4, 0, dB, 4, 0, dC, 4, 1, lg.GEMM_F32) == \
        lg.GEMM_ERR_UNSUPPORTED
