"""Python binding of libgemm (include/gemm.h): argument marshalling only.

Every function here has the name and the arguments of the C entry point it
wraps; pointers may be given as integers or as objects with ``data_ptr()``
(torch tensors), streams as integers, ``torch.cuda.Stream`` objects or None
(the current torch stream). All work runs in the CUDA kernels of
``libgemm.so``; there is no other code path: if the library is missing,
``load()`` raises.

    C[m][n] = sum_k A(m, k) * B(n, k)      (A is M x K, B is N x K)

as in the CuTe DSL Ampere SGEMM example (reference check "mk,nk->mn") and the
CK Tile practice GEMM. See include/gemm.h for layouts, types and status codes.
"""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgemm.so")

# enums of include/gemm.h
GEMM_MAJOR_K, GEMM_MAJOR_MN = 0, 1
GEMM_F32, GEMM_F16_F32, GEMM_BF16_F32, GEMM_F16_F16, GEMM_BF16_BF16 = 0, 1, 2, 3, 4
GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_CUDA, GEMM_ERR_TIMEOUT = \
    0, -1, -2, -3, -4
GEMM_OPT_WAIT_LIMIT_NS, GEMM_OPT_TC_CTA_GROUP, GEMM_OPT_TC_FAULT_INJECT = 1, 2, 3
GEMM_OPT_SIMT_CONFIG, GEMM_OPT_SIMT_TRANSPOSE, GEMM_OPT_TC_STORE = 4, 5, 6
GEMM_OPT_TC_MULTICAST, GEMM_OPT_SOFTMAX_FAULT_INJECT, GEMM_OPT_SIMT_SPLIT_TAIL = 7, 8, 9
GEMM_OPT_TC_SCHEDULER, GEMM_OPT_SIMT_FAULT_INJECT = 10, 11
GEMM_OPT_TC_TILE_N, GEMM_OPT_TC_SPLIT_TAIL = 12, 13
GEMM_ACT_NONE, GEMM_ACT_RELU, GEMM_ACT_GELU = 0, 1, 2


class GemmTuning(ctypes.Structure):
    """struct gemm_tuning: the configuration gemm_tune chose."""
    _fields_ = [("simt_config", ctypes.c_int), ("simt_transpose", ctypes.c_int),
                ("tc_cta_group", ctypes.c_int), ("tc_multicast", ctypes.c_int),
                ("tc_store", ctypes.c_int), ("ms", ctypes.c_float), ("candidates", ctypes.c_int),
                ("tc_scheduler", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class GemmEpilogue(ctypes.Structure):
    """struct gemm_epilogue: D = act(alpha * A B^T + beta * C + bias)."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("bias", ctypes.c_void_p), ("activation", ctypes.c_int)]

# storage type of A/B and of C per dtype
IN_TYPE = {GEMM_F32: "f32", GEMM_F16_F32: "f16", GEMM_BF16_F32: "bf16",
           GEMM_F16_F16: "f16", GEMM_BF16_BF16: "bf16"}
OUT_TYPE = {GEMM_F32: "f32", GEMM_F16_F32: "f32", GEMM_BF16_F32: "f32",
            GEMM_F16_F16: "f16", GEMM_BF16_BF16: "bf16"}

EXPORTS = ("gemm", "gemm_ex", "gemm_host", "gemm_noalloc", "gemm_tune", "gemm_tune_reset",
           "softmax_rows", "gemm_strerror", "gemm_check_device_error", "gemm_device_checks",
           "gemm_release_workspace", "gemm_launch_count", "gemm_set_option", "gemm_get_option")

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str = "gemm"):
        self.status = status
        super().__init__(f"{where}: status {status} ({gemm_strerror(status)})")


def load(path: str = LIB_PATH):
    """Load libgemm.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(
                f"libgemm.so not found at {path}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        sig = [i64, i64, i64, vp, i64, ci, vp, i64, ci, vp, i64, ci, ci, vp]
        for name in ("gemm", "gemm_host", "gemm_noalloc"):
            f = getattr(lib, name)
            f.restype, f.argtypes = ci, sig
        lib.gemm_ex.restype = ci
        lib.gemm_ex.argtypes = sig[:-1] + [ctypes.POINTER(GemmEpilogue), vp]
        lib.gemm_tune.restype = ci
        lib.gemm_tune.argtypes = sig[:-1] + [ci, vp, ctypes.POINTER(GemmTuning)]
        lib.gemm_tune_reset.restype, lib.gemm_tune_reset.argtypes = None, []
        lib.softmax_rows.restype = ci
        lib.softmax_rows.argtypes = [i64, i64, vp, i64, vp, i64, vp]
        lib.gemm_strerror.restype, lib.gemm_strerror.argtypes = ctypes.c_char_p, [ci]
        lib.gemm_check_device_error.restype = ci
        lib.gemm_check_device_error.argtypes = [vp]
        lib.gemm_device_checks.restype = ci
        lib.gemm_device_checks.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
        lib.gemm_release_workspace.restype, lib.gemm_release_workspace.argtypes = None, []
        lib.gemm_launch_count.restype, lib.gemm_launch_count.argtypes = ctypes.c_uint64, []
        lib.gemm_set_option.restype, lib.gemm_set_option.argtypes = ci, [ci, i64]
        lib.gemm_get_option.restype, lib.gemm_get_option.argtypes = i64, [ci]
        _lib = lib
        return lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):  # numpy array (host buffers for gemm_host)
        return int(x.ctypes.data)
    raise TypeError(f"cannot take a pointer of {type(x).__name__}")


def _stream(s) -> int:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return int(torch.cuda.current_stream().cuda_stream)
        except ImportError:
            pass
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def gemm(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype, stream=None) -> int:
    """C = A * B^T on device buffers; returns the gemm_status."""
    return load().gemm(M, N, K, _ptr(A), lda, a_major, _ptr(B), ldb, b_major, _ptr(C), ldc,
                       c_major, dtype, _stream(stream))


def gemm_ex(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype,
            alpha=1.0, beta=0.0, bias=None, activation=GEMM_ACT_NONE, stream=None) -> int:
    """C = act(alpha * A B^T + beta * C + bias[n]); see include/gemm.h."""
    epi = GemmEpilogue(alpha, beta, _ptr(bias) or None, activation)
    return load().gemm_ex(M, N, K, _ptr(A), lda, a_major, _ptr(B), ldb, b_major, _ptr(C), ldc,
                          c_major, dtype, ctypes.byref(epi), _stream(stream))


def gemm_host(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype,
              stream=None) -> int:
    """The same product on host buffers (copies inside, on `stream`)."""
    return load().gemm_host(M, N, K, _ptr(A), lda, a_major, _ptr(B), ldb, b_major, _ptr(C),
                            ldc, c_major, dtype, _stream(stream))


def gemm_noalloc(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype,
                 stream=None) -> int:
    """The 16-bit product with no device allocation (fixed 32 MiB repack
    scratch inside the library); see include/gemm.h."""
    return load().gemm_noalloc(M, N, K, _ptr(A), lda, a_major, _ptr(B), ldb, b_major, _ptr(C),
                               ldc, c_major, dtype, _stream(stream))


def gemm_tune(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype,
              iterations=5, stream=None):
    """Measure every configuration for this problem, record the fastest;
    returns (status, dict of the chosen configuration)."""
    t = GemmTuning()
    rc = load().gemm_tune(M, N, K, _ptr(A), lda, a_major, _ptr(B), ldb, b_major, _ptr(C), ldc,
                          c_major, dtype, iterations, _stream(stream), ctypes.byref(t))
    return rc, t.as_dict()


def gemm_tune_reset() -> None:
    load().gemm_tune_reset()


def softmax_rows(M, N, x, ldx, y, ldy, stream=None) -> int:
    """Row softmax of an fp32 matrix over thread-block clusters; see gemm.h."""
    return load().softmax_rows(M, N, _ptr(x), ldx, _ptr(y), ldy, _stream(stream))


def gemm_strerror(status: int) -> str:
    return load().gemm_strerror(status).decode()


def gemm_check_device_error(stream=None) -> int:
    return load().gemm_check_device_error(_stream(stream))


def gemm_device_checks(stream=None):
    """(status, first failed device-side check or 0); GEMM_ERR_UNSUPPORTED in a
    library built without the checks."""
    first = ctypes.c_uint64(0)
    rc = load().gemm_device_checks(_stream(stream), ctypes.byref(first))
    return rc, int(first.value)


def gemm_release_workspace() -> None:
    load().gemm_release_workspace()


def gemm_launch_count() -> int:
    return int(load().gemm_launch_count())


def gemm_set_option(option: int, value: int) -> int:
    return load().gemm_set_option(option, value)


def gemm_get_option(option: int) -> int:
    return int(load().gemm_get_option(option))


def check(status: int, where: str = "gemm") -> None:
    """Raise GemmError for a non-zero status."""
    if status != GEMM_OK:
        raise GemmError(status, where)
