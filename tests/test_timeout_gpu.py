"""Failure detection on the GPU without a fault: the tensor-core kernel's
pipeline waits are time-bounded. With the test hook GEMM_OPT_TC_FAULT_INJECT
the epilogue waits on a barrier that nothing completes; the wait must run
out after GEMM_OPT_WAIT_LIMIT_NS, the kernel must wind down (the MMA and
producer roles see the error word and stop, in-flight work drains, TMEM is
released), gemm_check_device_error must report GEMM_ERR_TIMEOUT once, and the
device must stay usable for correct GEMMs afterwards. The same holds for
softmax_rows' cluster exchange (GEMM_OPT_SOFTMAX_FAULT_INJECT: one CTA
withholds its partial, so its row's CTAs wait out the limit)."""

import numpy as np
import pytest

import datagen
import dense_gemm_06_gb300 as lg
import oracle
from gpu_util import check_full, make_operands, run_device_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


@pytest.mark.parametrize("scheduler", [1, 2])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_stalled_wait_times_out_and_device_recovers(cta_group, scheduler):
    import torch
    n, k = 4096, 512  # >= 3 tiles per CTA pair: the MMA role also blocks
    dA = torch.zeros(n * k, dtype=torch.int16, device="cuda")
    dB = torch.zeros(n * k, dtype=torch.int16, device="cuda")
    dC = torch.zeros(n * n, dtype=torch.int16, device="cuda")
    assert lg.gemm_check_device_error() == lg.GEMM_OK
    saved = {o: lg.gemm_get_option(o) for o in (lg.GEMM_OPT_WAIT_LIMIT_NS,
                                                lg.GEMM_OPT_TC_FAULT_INJECT,
                                                lg.GEMM_OPT_TC_CTA_GROUP,
                                                lg.GEMM_OPT_TC_SCHEDULER)}
    try:
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_WAIT_LIMIT_NS, 20_000_000))
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_CTA_GROUP, cta_group))
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_SCHEDULER, scheduler))
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_FAULT_INJECT, 1))
        rc = lg.gemm(n, n, k, dA, k, 0, dB, k, 0, dC, n, 1, lg.GEMM_BF16_BF16)
        assert rc == lg.GEMM_OK  # asynchronous: the timeout is reported later
        assert lg.gemm_check_device_error() == lg.GEMM_ERR_TIMEOUT
        assert lg.gemm_check_device_error() == lg.GEMM_OK  # the word was cleared
    finally:
        for o, v in saved.items():
            lg.gemm_set_option(o, v)
    # the context is intact: a normal GEMM on both paths is still exact
    for dtype in (lg.GEMM_F16_F32, lg.GEMM_F32):
        A, lda, B, ldb = make_operands(300, 520, 200, dtype, 0, 1, "int", 3)
        C = run_device_gemm(300, 520, 200, dtype, A, lda, 0, B, ldb, 1, cta_group=cta_group)
        check_full(C, 300, 520, 200, dtype, A, lda, 0, B, ldb, 1, exact=True,
                   what=f"after timeout (cg={cta_group})")


def test_stalled_ffma_tma_wait_times_out_and_device_recovers():
    # FFMA configuration 9: with GEMM_OPT_SIMT_FAULT_INJECT the first CTA
    # never loads its second k-tile, so its waits for that tile run out
    import torch
    M, N, K = 512, 512, 256
    dA = torch.zeros(K * M, dtype=torch.float32, device="cuda")
    dB = torch.zeros(K * N, dtype=torch.float32, device="cuda")
    dC = torch.zeros(M * N, dtype=torch.float32, device="cuda")
    assert lg.gemm_check_device_error() == lg.GEMM_OK
    saved = {o: lg.gemm_get_option(o) for o in (lg.GEMM_OPT_WAIT_LIMIT_NS,
                                                lg.GEMM_OPT_SIMT_FAULT_INJECT,
                                                lg.GEMM_OPT_SIMT_CONFIG)}
    try:
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_WAIT_LIMIT_NS, 20_000_000))
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, 9))
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_FAULT_INJECT, 1))
        rc = lg.gemm(M, N, K, dA, M, 1, dB, N, 1, dC, N, 1, lg.GEMM_F32)
        assert rc == lg.GEMM_OK  # asynchronous: the timeout is reported later
        assert lg.gemm_check_device_error() == lg.GEMM_ERR_TIMEOUT
        assert lg.gemm_check_device_error() == lg.GEMM_OK
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_FAULT_INJECT, 0))
        # the context is intact: the same kernel is exact again
        A, lda, B, ldb = make_operands(300, 520, 200, lg.GEMM_F32, 1, 1, "int", 4)
        C = run_device_gemm(300, 520, 200, lg.GEMM_F32, A, lda, 1, B, ldb, 1)
        check_full(C, 300, 520, 200, lg.GEMM_F32, A, lda, 1, B, ldb, 1, exact=True,
                   what="FFMA configuration 9 after a timeout")
    finally:
        for o, v in saved.items():
            lg.gemm_set_option(o, v)


def test_withheld_softmax_partial_times_out_and_device_recovers():
    import torch
    M, N = 6, 65536  # aligned rows of 65536 columns: clusters of 4 CTAs
    x = datagen.logical(M, N, dtype="f32", dist="normal", seed=11).astype(np.float32)
    dx = torch.from_numpy(x).cuda()
    dy = torch.empty_like(dx)
    assert lg.gemm_check_device_error() == lg.GEMM_OK
    saved = {o: lg.gemm_get_option(o) for o in (lg.GEMM_OPT_WAIT_LIMIT_NS,
                                                lg.GEMM_OPT_SOFTMAX_FAULT_INJECT)}
    try:
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_WAIT_LIMIT_NS, 20_000_000))
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_SOFTMAX_FAULT_INJECT, 1))
        assert lg.softmax_rows(M, N, dx, N, dy, N) == lg.GEMM_OK
        assert lg.gemm_check_device_error() == lg.GEMM_ERR_TIMEOUT
        assert lg.gemm_check_device_error() == lg.GEMM_OK
    finally:
        for o, v in saved.items():
            lg.gemm_set_option(o, v)
    # the context is intact and the exchange works again
    lg.check(lg.softmax_rows(M, N, dx, N, dy, N), "softmax_rows")
    lg.check(lg.gemm_check_device_error(), "device error word")
    y = dy.cpu().numpy().astype(np.float64)
    y_ref = oracle.softmax_ref(M, N, x.ravel(), N)
    assert np.all(np.abs(y - y_ref) <= 1e-5 * y_ref + 1e-30)


def _gemm_without_check(M, N, K, dtype, A, lda, am, B, ldb, bm):
    """gemm() through the C ABI, C read back WITHOUT gemm_check_device_error."""
    import torch
    from gpu_util import CBuffer, to_device
    cbuf = CBuffer(M, N, 1, N, lg.OUT_TYPE[dtype])
    lg.check(lg.gemm(M, N, K, to_device(A), lda, am, to_device(B), ldb, bm, cbuf.ptr(), N, 1,
                     dtype), "gemm")
    torch.cuda.synchronize()
    return cbuf.read()


@pytest.mark.parametrize("kernel", ["tcgen05", "ffma_tma"])
def test_timeout_is_confined_to_its_launch(kernel):
    # A wait of one launch runs out; the next launch -- made while the error
    # word still records that timeout (nobody has called
    # gemm_check_device_error) -- must run to the end and be exact, and the
    # check afterwards reports exactly one timeout.
    import torch
    hook = lg.GEMM_OPT_TC_FAULT_INJECT if kernel == "tcgen05" else lg.GEMM_OPT_SIMT_FAULT_INJECT
    saved = {o: lg.gemm_get_option(o) for o in (lg.GEMM_OPT_WAIT_LIMIT_NS, hook,
                                                lg.GEMM_OPT_SIMT_CONFIG)}
    assert lg.gemm_check_device_error() == lg.GEMM_OK
    try:
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_WAIT_LIMIT_NS, 20_000_000))
        if kernel == "tcgen05":
            n, k = 4096, 512
            dA = torch.zeros(n * k, dtype=torch.int16, device="cuda")
            dB = torch.zeros(n * k, dtype=torch.int16, device="cuda")
            dC = torch.zeros(n * n, dtype=torch.int16, device="cuda")
            lg.check(lg.gemm_set_option(hook, 1))
            assert lg.gemm(n, n, k, dA, k, 0, dB, k, 0, dC, n, 1, lg.GEMM_BF16_BF16) == lg.GEMM_OK
            dtype = lg.GEMM_F16_F32
        else:
            M, N, K = 512, 512, 256
            dA = torch.zeros(K * M, dtype=torch.float32, device="cuda")
            dB = torch.zeros(K * N, dtype=torch.float32, device="cuda")
            dC = torch.zeros(M * N, dtype=torch.float32, device="cuda")
            lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, 9))
            lg.check(lg.gemm_set_option(hook, 1))
            assert lg.gemm(M, N, K, dA, M, 1, dB, N, 1, dC, N, 1, lg.GEMM_F32) == lg.GEMM_OK
            dtype = lg.GEMM_F32
        torch.cuda.synchronize()  # the first launch has timed out and exited
        lg.check(lg.gemm_set_option(hook, 0))
        am = 0 if kernel == "tcgen05" else 1
        A, lda, B, ldb = make_operands(600, 520, 300, dtype, am, 1, "int", 5)
        C = _gemm_without_check(600, 520, 300, dtype, A, lda, am, B, ldb, 1)
        check_full(C, 600, 520, 300, dtype, A, lda, am, B, ldb, 1, exact=True,
                   what=f"{kernel} launch after another launch's timeout")
        assert lg.gemm_check_device_error() == lg.GEMM_ERR_TIMEOUT  # the first launch's
        assert lg.gemm_check_device_error() == lg.GEMM_OK
    finally:
        for o, v in saved.items():
            lg.gemm_set_option(o, v)
