"""gemm_tune: per-problem configuration selection (the pages' autotune
utilities done natively). It must measure every configuration valid for the
problem, leave a correct product in C, record a valid choice that later
gemm() calls on the same problem use, and forget it on gemm_tune_reset."""

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
    lg.gemm_tune_reset()
    yield
    lg.gemm_tune_reset()


@pytest.mark.parametrize("dtype,am,bm,cm,ldc_pad,expect", [
    (lg.GEMM_F32, 0, 0, 1, 0, 18),        # 9 tile configs x {as is, transposed}
    (lg.GEMM_F32, 1, 1, 1, 0, 9),         # MN-major operands: nothing to transpose
    (lg.GEMM_BF16_BF16, 0, 1, 1, 0, 8),   # 4 CTA modes / schedulers x 2 store paths
    (lg.GEMM_F16_F32, 1, 0, 0, 1, 4),     # misaligned C: st.global only
])
def test_tune_records_a_valid_choice(dtype, am, bm, cm, ldc_pad, expect):
    import torch
    M, N, K = 1000, 704, 600  # 704 * 2 bytes: 16-byte aligned rows for every C type
    A, lda, B, ldb = make_operands(M, N, K, dtype, am, bm, "int", 31)
    dA, dB = to_device(A), to_device(B)
    ldc = (N if cm == 1 else M) + ldc_pad
    cbuf = CBuffer(M, N, cm, ldc, lg.OUT_TYPE[dtype])
    rc, t = lg.gemm_tune(M, N, K, dA, lda, am, dB, ldb, bm, cbuf.ptr(), ldc, cm, dtype,
                         iterations=2)
    assert rc == lg.GEMM_OK and t["candidates"] == expect and t["ms"] > 0
    if dtype == lg.GEMM_F32:
        assert 1 <= t["simt_config"] <= 9 and t["simt_transpose"] in (1, 2)
    else:
        # the operand-multicast variant is never a tuning candidate
        assert (t["tc_cta_group"], t["tc_multicast"], t["tc_scheduler"]) in (
            (1, 1, 1), (1, 1, 2), (2, 1, 1), (2, 1, 2))
        assert t["tc_store"] in ((1,) if ldc_pad else (0, 1))
    torch.cuda.synchronize()
    exact = lg.OUT_TYPE[dtype] == "f32"
    # the tuned runs leave the product in C
    check_full(cbuf.read(), M, N, K, dtype, A, lda, am, B, ldb, bm, exact=exact,
               what="after gemm_tune")
    # a later gemm() on the same problem runs the recorded configuration
    cbuf2 = CBuffer(M, N, cm, ldc, lg.OUT_TYPE[dtype])
    lg.check(lg.gemm(M, N, K, dA, lda, am, dB, ldb, bm, cbuf2.ptr(), ldc, cm, dtype))
    lg.check(lg.gemm_check_device_error())
    torch.cuda.synchronize()
    check_full(cbuf2.read(), M, N, K, dtype, A, lda, am, B, ldb, bm, exact=exact,
               what="gemm after gemm_tune")


def test_tune_nothing_to_run():
    rc, t = lg.gemm_tune(0, 5, 5, 0, 5, 0, 0, 5, 0, 0, 5, 1, lg.GEMM_F32)
    assert rc == lg.GEMM_OK and t["candidates"] == 0
    assert lg.gemm_tune(-1, 5, 5, 0, 5, 0, 0, 5, 0, 0, 5, 1, lg.GEMM_F32)[0] == \
        lg.GEMM_ERR_INVALID_ARG
