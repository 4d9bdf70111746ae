"""The C-ABI boundary (CPU part): the library loads, exports every function
include/gemm.h declares, and rejects bad arguments on the host before any
CUDA call. Host-side checks follow the validation of the Gluon Multi-CTA
tutorial's matmul_multicta wrapper (shape/dtype checks before launching),
reported as status codes."""

import ctypes
import os
import re

import pytest

import dense_gemm_06_gb300 as lg
from dense_gemm_06_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return lg.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                      text, flags=re.M)


def test_header_declares_the_binding_names():
    assert sorted(declared_functions()) == sorted(lg.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_enums_match_header():
    text = open(HEADER).read()
    for name in ("GEMM_MAJOR_K", "GEMM_MAJOR_MN", "GEMM_F32", "GEMM_F16_F32", "GEMM_BF16_F32",
                 "GEMM_F16_F16", "GEMM_BF16_BF16", "GEMM_OK", "GEMM_ERR_INVALID_ARG",
                 "GEMM_ERR_UNSUPPORTED", "GEMM_ERR_CUDA", "GEMM_ERR_TIMEOUT",
                 "GEMM_OPT_WAIT_LIMIT_NS", "GEMM_OPT_TC_CTA_GROUP", "GEMM_OPT_TC_FAULT_INJECT",
                 "GEMM_OPT_SIMT_CONFIG", "GEMM_OPT_SIMT_TRANSPOSE", "GEMM_OPT_TC_STORE",
                 "GEMM_OPT_TC_MULTICAST", "GEMM_OPT_SOFTMAX_FAULT_INJECT",
                 "GEMM_OPT_SIMT_SPLIT_TAIL", "GEMM_OPT_TC_SCHEDULER",
                 "GEMM_OPT_SIMT_FAULT_INJECT", "GEMM_ACT_NONE",
                 "GEMM_ACT_RELU", "GEMM_ACT_GELU"):
        m = re.search(rf"\b{name}\s*=\s*(-?\d+)", text)
        assert m, name
        assert int(m.group(1)) == getattr(lg, name), name


P = 0x10000  # a fake, 16-byte aligned address: validation never dereferences


def call(M=4, N=4, K=4, A=P, lda=None, am=0, B=P, ldb=None, bm=0, C=P, ldc=None, cm=1,
         dtype=lg.GEMM_F32):
    lda = lda if lda is not None else (K if am == 0 else M)
    ldb = ldb if ldb is not None else (K if bm == 0 else N)
    ldc = ldc if ldc is not None else (N if cm == 1 else M)
    return lg.gemm(M, N, K, A, lda, am, B, ldb, bm, C, ldc, cm, dtype, 0)


@pytest.mark.parametrize("kw", [
    dict(M=-1), dict(N=-1), dict(K=-1), dict(M=1 << 31), dict(dtype=5), dict(dtype=-1),
    dict(am=2), dict(bm=-1), dict(cm=3),
    dict(A=0), dict(B=0), dict(C=0),
    dict(lda=3), dict(ldb=3), dict(ldc=3),
    dict(am=1, lda=3), dict(bm=1, ldb=3), dict(cm=0, ldc=3),
    dict(A=P + 2), dict(B=P + 1, dtype=lg.GEMM_BF16_F32), dict(C=P + 2),
    dict(C=P + 2, dtype=lg.GEMM_F16_F32), dict(M=1 << 30, lda=1 << 62),
])
def test_invalid_arguments_rejected_on_host(lib, kw):
    assert call(**kw) == lg.GEMM_ERR_INVALID_ARG


def test_valid_element_alignment_passes_validation(lib):
    # 2-byte aligned 16-bit operands and odd leading dimensions are legal; with
    # no usable sm_103 device the call then stops at the device check.
    rc = call(A=P + 2, B=P + 6, lda=7, ldb=5, C=P + 4, ldc=9, dtype=lg.GEMM_F16_F32)
    assert rc in (lg.GEMM_ERR_UNSUPPORTED, lg.GEMM_OK) or rc == lg.GEMM_ERR_CUDA


def test_gemm_ex_host_checks(lib):
    assert lg.gemm_ex(4, 4, 4, P, 4, 0, P, 4, 0, P, 4, 1, lg.GEMM_F32, activation=3) == \
        lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_ex(4, 4, 4, P, 4, 0, P, 4, 0, P, 4, 1, lg.GEMM_F32, bias=P + 2) == \
        lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_ex(-1, 4, 4, P, 4, 0, P, 4, 0, P, 4, 1, lg.GEMM_F32, beta=1.0) == \
        lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_ex(0, 4, 4, P, 4, 0, P, 4, 0, P, 4, 1, lg.GEMM_F32, beta=1.0) == lg.GEMM_OK


def test_softmax_host_checks(lib):
    assert lg.softmax_rows(-1, 4, P, 4, P, 4) == lg.GEMM_ERR_INVALID_ARG
    assert lg.softmax_rows(4, 4, 0, 4, P, 4) == lg.GEMM_ERR_INVALID_ARG
    assert lg.softmax_rows(4, 4, P, 3, P, 4) == lg.GEMM_ERR_INVALID_ARG
    assert lg.softmax_rows(4, 4, P + 2, 4, P, 4) == lg.GEMM_ERR_INVALID_ARG
    assert lg.softmax_rows(0, 4, 0, 4, 0, 4) == lg.GEMM_OK
    assert lg.softmax_rows(2, 524289, P, 524289, P, 524289) == lg.GEMM_ERR_UNSUPPORTED


def test_degenerate_sizes_need_no_device(lib):
    assert call(M=0) == lg.GEMM_OK
    assert call(N=0, C=0) == lg.GEMM_OK          # nothing addressed: C may be NULL
    assert call(M=0, A=0, B=0, C=0) == lg.GEMM_OK


def test_k_zero_needs_no_operands(lib):
    rc = call(K=0, A=0, B=0, lda=0, ldb=0)
    assert rc != lg.GEMM_ERR_INVALID_ARG


def test_no_gpu_reports_unsupported(lib):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    assert call() == lg.GEMM_ERR_UNSUPPORTED
    assert lg.gemm_host(4, 4, 4, P, 4, 0, P, 4, 0, P, 4, 1, lg.GEMM_F32, 0) == \
        lg.GEMM_ERR_UNSUPPORTED
    assert lg.gemm_check_device_error(0) == lg.GEMM_ERR_UNSUPPORTED
    lg.gemm_release_workspace()  # harmless without a device


def test_strerror_and_options(lib):
    for s in (0, -1, -2, -3, -4, 7):
        assert isinstance(lg.gemm_strerror(s), str) and lg.gemm_strerror(s)
    assert lg.gemm_strerror(-4) != lg.gemm_strerror(0)
    assert lg.gemm_get_option(lg.GEMM_OPT_WAIT_LIMIT_NS) == 1_000_000_000
    assert lg.gemm_set_option(lg.GEMM_OPT_WAIT_LIMIT_NS, 5_000_000) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_WAIT_LIMIT_NS) == 5_000_000
    assert lg.gemm_set_option(lg.GEMM_OPT_WAIT_LIMIT_NS, 0) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_WAIT_LIMIT_NS) == 1_000_000_000
    assert lg.gemm_set_option(lg.GEMM_OPT_WAIT_LIMIT_NS, -5) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_CTA_GROUP, 3) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_FAULT_INJECT, 2) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_set_option(99, 0) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_get_option(99) == -1
    assert lg.gemm_get_option(lg.GEMM_OPT_TC_CTA_GROUP) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_TC_FAULT_INJECT) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_SIMT_CONFIG) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, 10) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, 9) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, 0) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_SIMT_TRANSPOSE) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_TRANSPOSE, 3) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_get_option(lg.GEMM_OPT_TC_STORE) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_STORE, 2) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_get_option(lg.GEMM_OPT_TC_MULTICAST) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_MULTICAST, 3) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_get_option(lg.GEMM_OPT_SOFTMAX_FAULT_INJECT) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_SOFTMAX_FAULT_INJECT, 2) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_get_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 4) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 3) == 0   # stream-K (tests)
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 2) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL) == 2
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 0) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_TC_SCHEDULER) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_SCHEDULER, 3) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_get_option(lg.GEMM_OPT_SIMT_FAULT_INJECT) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_SIMT_FAULT_INJECT, 2) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_get_option(lg.GEMM_OPT_TC_TILE_N) == 0
    for bad in (32, 96, 512, -1):
        assert lg.gemm_set_option(lg.GEMM_OPT_TC_TILE_N, bad) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_TILE_N, 64) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_TC_TILE_N) == 64
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_TILE_N, 0) == 0
    assert lg.gemm_get_option(lg.GEMM_OPT_TC_SPLIT_TAIL) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_SPLIT_TAIL, 3) == lg.GEMM_ERR_INVALID_ARG
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_SPLIT_TAIL, 2) == 0
    assert lg.gemm_set_option(lg.GEMM_OPT_TC_SPLIT_TAIL, 0) == 0


def test_launch_count_unchanged_by_rejected_calls(lib):
    n = lg.gemm_launch_count()
    call(M=-1)
    call(M=0)
    assert lg.gemm_launch_count() == n


def test_missing_library_fails_loudly(tmp_path):
    import importlib
    mod = importlib.import_module("dense_gemm_06_gb300")
    with pytest.raises(ImportError):
        # a fresh loader pointed at a path with no library
        saved = mod._lib
        try:
            mod._lib = None
            mod.load(str(tmp_path / "libgemm.so"))
        finally:
            mod._lib = saved


def test_device_checks_absent_from_the_default_build(lib):
    # gemm_device_checks answers only in the debug build with device-side
    # checks; the default library says so without touching a device
    rc, first = lg.gemm_device_checks()
    assert rc == lg.GEMM_ERR_UNSUPPORTED and first == 0
