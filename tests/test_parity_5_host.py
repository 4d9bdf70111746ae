"""GPU parity of gemm_host (host buffers in and out) against the oracle.

Small problems run as one panel; large ones are cut into row panels of C
whose A rows (or columns) go in, compute and C rows come back on separate
copy streams, so the cases below cover one and several panels, every C
major, K- and MN-major A and B, padded leading dimensions, pinned and
pageable host memory, and K = 0. Integer-valued inputs: compared bit-exactly
(16-bit C: against round-to-nearest-even of C_ref)."""

import itertools

import numpy as np
import pytest

import datagen
import dense_gemm_06_gb300 as lg
import oracle
from gpu_util import decode, make_operands

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


NAN = {"f32": np.float32(np.nan), "f16": np.uint16(0x7E5A), "bf16": np.uint16(0x7FDA)}


def host_gemm(M, N, K, dtype, am, bm, cm, seed, pad=0, pinned=False):
    """Runs gemm_host; returns (logical C as float64, operands)."""
    import torch
    ot = lg.OUT_TYPE[dtype]
    A, lda, B, ldb = make_operands(M, N, K, dtype, am, bm, "int", seed, lda_pad=pad,
                                   ldb_pad=pad, lo=-3, hi=3)
    ldc = (N if cm == lg.GEMM_MAJOR_MN else M) + pad
    outer = M if cm == lg.GEMM_MAJOR_MN else N
    inner = N if cm == lg.GEMM_MAJOR_MN else M
    C = np.full(outer * ldc, NAN[ot], np.float32 if ot == "f32" else np.uint16)
    if pinned:
        tA, tB = torch.from_numpy(A.view(np.int16) if A.dtype == np.uint16 else A), \
            torch.from_numpy(B.view(np.int16) if B.dtype == np.uint16 else B)
        tC = torch.from_numpy(C.view(np.int16) if C.dtype == np.uint16 else C)
        hA, hB, hC = tA.pin_memory(), tB.pin_memory(), tC.pin_memory()
    else:
        hA, hB, hC = A, B, C
    lg.check(lg.gemm_host(M, N, K, hA if K else 0, lda, am, hB if K else 0, ldb, bm, hC, ldc, cm,
                          dtype), "gemm_host")
    lg.check(lg.gemm_check_device_error(), "device error word")
    torch.cuda.synchronize()
    raw = hC.numpy() if pinned else hC
    raw = raw.view(np.float32) if ot == "f32" else raw.view(np.uint16)
    grid = raw.reshape(outer, ldc)
    if ldc > inner:  # padding of C is never written
        assert np.array_equal(grid[:, inner:].view(np.uint8),
                              np.full_like(grid[:, inner:], NAN[ot]).view(np.uint8))
    vals = decode(np.ascontiguousarray(grid[:, :inner]), ot)
    Cl = vals if cm == lg.GEMM_MAJOR_MN else vals.T.copy()
    return Cl, A, lda, B, ldb


def rne(x, t):
    if t == "f16":
        return x.astype(np.float16).astype(np.float64)
    if t == "bf16":
        bits = datagen.f32_to_bf16_bits(x.astype(np.float32))
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x


@pytest.mark.parametrize("dtype", [lg.GEMM_F32, lg.GEMM_F16_F32, lg.GEMM_BF16_BF16])
@pytest.mark.parametrize("am,bm,cm", list(itertools.product((0, 1), (0, 1), (0, 1))))
def test_host_one_panel(dtype, am, bm, cm):
    M, N, K = 300, 260, 130
    C, A, lda, B, ldb = host_gemm(M, N, K, dtype, am, bm, cm, seed=50, pad=(am + cm) % 2 * 3)
    it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
    C_ref, S = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, bm, it)
    assert np.array_equal(C, rne(C_ref, ot)), f"{M}x{N}x{K} dtype={dtype} {am}{bm}{cm}"


@pytest.mark.parametrize("dtype,M,N,K", [(lg.GEMM_F32, 4096, 2048, 2048),
                                         (lg.GEMM_BF16_F32, 8192, 2048, 1024),
                                         (lg.GEMM_F16_F16, 8192, 2048, 1024),
                                         (lg.GEMM_F32, 2560, 8192, 1024),
                                         (lg.GEMM_BF16_BF16, 8192, 4096, 1024)])
@pytest.mark.parametrize("am,cm", [(0, 1), (1, 1), (0, 0), (1, 0)])
def test_host_several_panels(dtype, M, N, K, am, cm):
    # M * N * K >= 1e10: row panels of C in whole waves of tiles
    C, A, lda, B, ldb = host_gemm(M, N, K, dtype, am, 1 - am, cm, seed=51, pinned=(am == 0))
    it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
    rows = datagen.sample_indices(M, 128, seed=52, stream=101)
    cols = datagen.sample_indices(N, 128, seed=52, stream=102)
    Cr, Sr = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, 1 - am, it, rows=rows)
    assert np.array_equal(C[rows, :], rne(Cr, ot)), "sampled rows"
    Cc, Sc = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, 1 - am, it, cols=cols)
    assert np.array_equal(C[:, cols], rne(Cc, ot)), "sampled cols"
    # panel boundaries: every row near a multiple of 128 is checked in full
    edge = np.unique(np.clip(np.concatenate([np.arange(128, M, 128) - 1,
                                             np.arange(128, M, 128)]), 0, M - 1))[::7]
    Ce, _ = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, 1 - am, it, rows=edge)
    assert np.array_equal(C[edge, :], rne(Ce, ot)), "rows at tile boundaries"


def test_host_k_zero_writes_zero():
    C, *_ = host_gemm(70, 50, 0, lg.GEMM_F32, 0, 0, 1, seed=53, pad=2)
    assert np.all(C == 0.0)
