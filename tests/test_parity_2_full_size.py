"""GPU parity on the full-size workloads, in the launch configuration the
benchmark times (default options: the 2-CTA tensor-core kernel, the FFMA
kernel for fp32).

* 1024 x 512 x 256 fp16 integers in [-5, 5] (A, B K-major) -> fp32 C
   row-major: the CK Tile practice GEMM's "Problem Size Configuration" and
   integer fill; bit-exact against the full oracle.
* 2048^3 fp32 SGEMM, A M-major, B N-major, C N-major, U[-1, 1]: the CuTe
   Ampere SGEMM example's documented layout (a_major m, b_major n, c_major
   n); full oracle, |C - C_ref| <= 1e-4 * S.
* 8192^3 fp32 SGEMM over all four A/B majors, N(0, 1): the CuTe example's
   ncu recipe size; 256 seeded rows and 256 seeded columns (plus the first
   and last) against the oracle.
* 8192^3 bf16 -> bf16 (A, B K-major), N(0, 1) rounded to bf16: the Gluon
   Multi-CTA tutorial's benchmark size; sampled rows/columns, 1 bf16 ulp +
   1e-4 * S.
* 4095 x 3071 x 1037 (A K-major, B N-major, packed: lda 1037, ldb 3071,
   ldc 3071, none 16-byte multiples) and 16384 x 256 x 8192, fp16 integers
   in [-3, 3] -> fp32; bit-exact against the full oracle.

Seeds: 1025 (1024 x 512 x 256), 1026 (2048^3), 1027 (8192^3 fp32), 1028
(8192^3 bf16), 1029 (4095 x 3071 x 1037), 1030 (16384 x 256 x 8192).
"""

import numpy as np
import pytest

import datagen
import dense_gemm_06_gb300 as lg
import oracle
from gpu_util import check_full, check_sampled, decode, make_operands, run_device_gemm, to_device


def rne16(x: np.ndarray, t: str) -> np.ndarray:
    """Round exact (integer-valued) results to the 16-bit output type."""
    if t == "f16":
        return x.astype(np.float16).astype(np.float64)
    bits = datagen.f32_to_bf16_bits(x.astype(np.float32))
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


@pytest.mark.parametrize("cta_group", [0, 1])
def test_fp16_int_1024x512x256_bit_exact(cta_group):
    M, N, K = 1024, 512, 256
    A, lda, B, ldb = make_operands(M, N, K, lg.GEMM_F16_F32, 0, 0, "int", 1025)
    C = run_device_gemm(M, N, K, lg.GEMM_F16_F32, A, lda, 0, B, ldb, 0, cta_group=cta_group)
    check_full(C, M, N, K, lg.GEMM_F16_F32, A, lda, 0, B, ldb, 0, exact=True,
               what=f"1024x512x256 fp16 int (cg={cta_group})")


def test_fp32_2048_cubed_a_m_b_n():
    M = N = K = 2048
    A, lda, B, ldb = make_operands(M, N, K, lg.GEMM_F32, 1, 1, "pm1", 1026)
    C = run_device_gemm(M, N, K, lg.GEMM_F32, A, lda, 1, B, ldb, 1)
    check_full(C, M, N, K, lg.GEMM_F32, A, lda, 1, B, ldb, 1, exact=False, what="2048^3 fp32")


@pytest.fixture(scope="module")
def fp32_8192_logical():
    n = 8192
    LA = datagen.logical(n, n, dtype="f32", dist="normal", seed=1027, stream=0)
    LB = datagen.logical(n, n, dtype="f32", dist="normal", seed=1027, stream=1)
    return LA, LB


@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_fp32_8192_cubed_all_majors(fp32_8192_logical, am, bm):
    n = 8192
    LA, LB = fp32_8192_logical
    A = (LA if am == 0 else LA.T).copy().ravel()
    B = (LB if bm == 0 else LB.T).copy().ravel()
    C = run_device_gemm(n, n, n, lg.GEMM_F32, A, n, am, B, n, bm)
    check_sampled(C, n, n, n, lg.GEMM_F32, A, n, am, B, n, bm, exact=False,
                  what=f"8192^3 fp32 A{'KM'[am]} B{'KN'[bm]}", seed=1027)


@pytest.mark.parametrize("cta_group,multicast,scheduler",
                         [(0, 0, 0), (1, 0, 0), (2, 2, 0), (2, 1, 2), (1, 1, 2)])
def test_bf16_8192_cubed(cta_group, multicast, scheduler):
    n = 8192
    A, lda, B, ldb = make_operands(n, n, n, lg.GEMM_BF16_BF16, 0, 0, "normal", 1028)
    C = run_device_gemm(n, n, n, lg.GEMM_BF16_BF16, A, lda, 0, B, ldb, 0, cta_group=cta_group,
                        multicast=multicast, scheduler=scheduler)
    check_sampled(C, n, n, n, lg.GEMM_BF16_BF16, A, lda, 0, B, ldb, 0, exact=False,
                  what=f"8192^3 bf16 (cg={cta_group}, mc={multicast}, sched={scheduler})",
                  seed=1028)


@pytest.mark.parametrize("scheduler", [0, 2])
def test_fp16_int_4095x3071x1037_ragged_bit_exact(scheduler):
    M, N, K = 4095, 3071, 1037
    A, lda, B, ldb = make_operands(M, N, K, lg.GEMM_F16_F32, 0, 1, "int", 1029, lo=-3, hi=3)
    assert (lda, ldb) == (1037, 3071)
    C = run_device_gemm(M, N, K, lg.GEMM_F16_F32, A, lda, 0, B, ldb, 1, scheduler=scheduler)
    check_full(C, M, N, K, lg.GEMM_F16_F32, A, lda, 0, B, ldb, 1, exact=True, what="4095x3071x1037 fp16 int")


@pytest.mark.parametrize("scheduler", [0, 2])
def test_fp16_int_16384x256x8192_skinny_bit_exact(scheduler):
    M, N, K = 16384, 256, 8192
    A, lda, B, ldb = make_operands(M, N, K, lg.GEMM_F16_F32, 0, 1, "int", 1030, lo=-3, hi=3)
    C = run_device_gemm(M, N, K, lg.GEMM_F16_F32, A, lda, 0, B, ldb, 1, scheduler=scheduler)
    check_full(C, M, N, K, lg.GEMM_F16_F32, A, lda, 0, B, ldb, 1, exact=True, what="16384x256x8192 fp16 int")


@pytest.mark.parametrize("dtype,am,bm,cm", [(lg.GEMM_F32, 0, 1, 1), (lg.GEMM_BF16_BF16, 0, 0, 0)])
def test_c_beyond_4g_elements(dtype, am, bm, cm):
    # C with 70001 x 65537 > 2^32 elements (18.4 GB in fp32): every row offset
    # past 2^32 elements must be formed in 64 bits. Guard bands of 64 elements
    # on both sides of C must stay untouched; rows and columns are sampled
    # (the first and last included) and compared bit-exactly.
    import torch
    M, N, K = 70001, 65537, 40
    ot = lg.OUT_TYPE[dtype]
    A, lda, B, ldb = make_operands(M, N, K, dtype, am, bm, "int", 1040, lo=-3, hi=3)
    ldc = N if cm == 1 else M
    outer = M if cm == 1 else N
    tdt = torch.float32 if ot == "f32" else torch.int16
    canary = float("nan") if ot == "f32" else 0x7FDA
    dC = torch.full((outer * ldc + 128,), canary, dtype=tdt, device="cuda")
    esz = 4 if ot == "f32" else 2
    lg.check(lg.gemm(M, N, K, to_device(A), lda, am, to_device(B), ldb, bm,
                     int(dC.data_ptr()) + 64 * esz, ldc, cm, dtype), "gemm")
    lg.check(lg.gemm_check_device_error(), "device error word")
    torch.cuda.synchronize()
    guard = torch.cat([dC[:64], dC[-64:]]).cpu().numpy()
    if ot == "f32":
        assert np.all(np.isnan(guard)), "guard band written"
    else:
        assert np.all(guard.view(np.uint16) == 0x7FDA), "guard band written"
    body = dC[64:64 + outer * ldc].view(outer, ldc)
    it = lg.IN_TYPE[dtype]
    rows = datagen.sample_indices(M, 48, seed=1041, stream=101)
    cols = datagen.sample_indices(N, 48, seed=1041, stream=102)

    def logical(block):  # device block of storage -> logical float64
        raw = block.cpu().numpy()
        return decode(raw.view(np.float32) if ot == "f32" else raw.view(np.uint16), ot)

    if cm == 1:
        Cr = logical(body[torch.as_tensor(rows, device="cuda")])
        Cc = logical(body[:, torch.as_tensor(cols, device="cuda")])
    else:
        Cr = logical(body[:, torch.as_tensor(rows, device="cuda")]).T
        Cc = logical(body[torch.as_tensor(cols, device="cuda")]).T
    R, _ = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, bm, it, rows=rows)
    Cl, _ = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, bm, it, cols=cols)
    want_r, want_c = (R, Cl) if ot == "f32" else (rne16(R, ot), rne16(Cl, ot))
    assert np.array_equal(Cr, want_r), "sampled rows"
    assert np.array_equal(Cc, want_c), "sampled columns"
    del dC, body
    torch.cuda.empty_cache()
