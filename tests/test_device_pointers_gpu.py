"""Every device entry point takes memory of the current device only: host
pointers (pinned or pageable) are rejected with GEMM_ERR_INVALID_ARG on the
host, before any launch, whatever the kernel options -- including the
opt-in cluster-multicast variant, whose TMA loads must only ever address this
GPU's own memory."""

import numpy as np
import pytest

import dense_gemm_06_gb300 as lg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


@pytest.mark.parametrize("multicast", [0, 2])
def test_host_pointers_rejected_before_any_launch(multicast):
    import torch
    M = N = K = 512
    dev = {k: torch.zeros(M * K, dtype=torch.int16, device="cuda") for k in "ABC"}
    dev["C"] = torch.zeros(M * N, dtype=torch.float32, device="cuda")
    pinned = {k: torch.zeros_like(v, device="cpu").pin_memory() for k, v in dev.items()}
    pageable = {k: np.zeros(v.numel(), dtype=np.int16 if k != "C" else np.float32)
                for k, v in dev.items()}
    saved = lg.gemm_get_option(lg.GEMM_OPT_TC_MULTICAST)
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_MULTICAST, multicast))
    n0 = lg.gemm_launch_count()
    try:
        for host in (pinned, pageable):
            for bad in "ABC":
                ops = {k: (host[k] if k == bad else dev[k]) for k in "ABC"}
                args = (M, N, K, ops["A"], K, 0, ops["B"], K, 0, ops["C"], N, 1,
                        lg.GEMM_F16_F32)
                assert lg.gemm(*args) == lg.GEMM_ERR_INVALID_ARG, bad
                assert lg.gemm_ex(*args, alpha=2.0) == lg.GEMM_ERR_INVALID_ARG, bad
                assert lg.gemm_noalloc(*args) == lg.GEMM_ERR_INVALID_ARG, bad
                rc, _ = lg.gemm_tune(*args)
                assert rc == lg.GEMM_ERR_INVALID_ARG, bad
            # a host bias vector
            assert lg.gemm_ex(M, N, K, dev["A"], K, 0, dev["B"], K, 0, dev["C"], N, 1,
                              lg.GEMM_F16_F32, bias=host["C"]) == lg.GEMM_ERR_INVALID_ARG
            # fp32 inputs (the FFMA kernel) and the row softmax
            x = torch.zeros(M * N, dtype=torch.float32, device="cuda")
            assert lg.gemm(M, N, K, host["C"], K, 0, x, K, 0, dev["C"], N, 1,
                           lg.GEMM_F32) == lg.GEMM_ERR_INVALID_ARG
            assert lg.softmax_rows(M, N, host["C"], N, x, N) == lg.GEMM_ERR_INVALID_ARG
            assert lg.softmax_rows(M, N, x, N, host["C"], N) == lg.GEMM_ERR_INVALID_ARG
        assert lg.gemm_launch_count() == n0  # nothing was launched
        # device memory of this GPU is accepted
        lg.check(lg.gemm(M, N, K, dev["A"], K, 0, dev["B"], K, 0, dev["C"], N, 1,
                         lg.GEMM_F16_F32), "gemm")
        lg.check(lg.gemm_check_device_error(), "device error word")
        assert lg.gemm_launch_count() > n0
    finally:
        lg.gemm_set_option(lg.GEMM_OPT_TC_MULTICAST, saved)
