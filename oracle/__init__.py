"""CPU oracle for dense GEMM -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package. The CUDA
library never imports it and shares no code with it.

``gemm_ref`` returns ``C_ref`` and ``S`` (both float64) for a block of rows
and columns of ``C = A * B^T``:

    C_ref[m, n] = sum_k A(m, k) * B(n, k)      (fp64, ascending k)
    S[m, n]     = sum_k |A(m, k) * B(n, k)|

as the CuTe DSL Ampere SGEMM example's reference check defines the product
(``einsum("mk,nk->mn")`` in its ``run()``) and as the CK Tile practice GEMM's
"Result Verification" checks it with a CPU GEMM. The arithmetic is the plain C
triple loop in ``gemm_oracle.c``; this module only marshals buffers.

Pins: ``tests/test_oracle.py`` checks this oracle against exact rational
brute force, closed forms, identity/permutation/linearity/transpose
invariants and the element decoders against numpy on every bit pattern.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``liboracle.so`` (plain gcc, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_gemm.argtypes = [i64, i64, i64,
                                        p, i64, ctypes.c_int, ctypes.c_int,
                                        p, i64, ctypes.c_int, ctypes.c_int,
                                        p, i64, p, i64, p, p, ctypes.c_int]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f32_to_f64.restype = ctypes.c_double
            lib.oracle_f32_to_f64.argtypes = [ctypes.c_uint32]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_softmax_rows.restype = ctypes.c_int
            lib.oracle_softmax_rows.argtypes = [i64, i64, p, i64, p, i64]
            lib.oracle_epilogue.restype = ctypes.c_int
            lib.oracle_epilogue.argtypes = [i64, i64, p, p, i64, p, i64, ctypes.c_double,
                                            ctypes.c_double, p, i64, ctypes.c_int, ctypes.c_int,
                                            p, ctypes.c_int, p]
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle uses by default (online host cores)."""
    return _load().oracle_num_threads()


def decode(bits: int, dtype: str) -> float:
    """Exact value of one stored element (bits of an f32/f16/bf16)."""
    lib = _load()
    if dtype == "f16":
        return lib.oracle_f16_to_f64(bits)
    if dtype == "bf16":
        return lib.oracle_bf16_to_f64(bits)
    return lib.oracle_f32_to_f64(bits)


def _ptr(a):
    return None if a is None or a.size == 0 else a.ctypes.data


def gemm_ref(M: int, N: int, K: int,
             A: np.ndarray, lda: int, a_major: int, a_dtype: str,
             B: np.ndarray, ldb: int, b_major: int, b_dtype: str,
             rows=None, cols=None, threads: int = 0, with_s: bool = True):
    """(C_ref, S) of shape (len(rows), len(cols)); all rows/cols when None.

    ``A``/``B`` are flat storage arrays (float32, or uint16 bit patterns for
    f16/bf16) addressed as the C ABI does: A K-major ``A[m*lda+k]``, A M-major
    ``A[k*lda+m]``, B K-major ``B[n*ldb+k]``, B N-major ``B[k*ldb+n]``.
    """
    lib = _load()
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else len(r)
    nc = N if c is None else len(c)
    C = np.zeros((nr, nc), dtype=np.float64)
    S = np.zeros((nr, nc), dtype=np.float64) if with_s else None
    if nr == 0 or nc == 0:
        return C, S
    rc = lib.oracle_gemm(M, N, K,
                         _ptr(A), lda, a_major, DTYPES[a_dtype],
                         _ptr(B), ldb, b_major, DTYPES[b_dtype],
                         None if r is None else r.ctypes.data, nr,
                         None if c is None else c.ctypes.data, nc,
                         _ptr(C), _ptr(S) if with_s else None, threads)
    if rc != 0:
        raise ValueError(f"oracle_gemm rejected the arguments (status {rc})")
    return C, S


ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}


def epilogue_ref(M: int, N: int, C_ref: np.ndarray, alpha: float, beta: float,
                 C_in=None, ldc: int = 0, c_major: int = 1, c_dtype: str = "f32",
                 bias=None, act: str = "none", rows=None, cols=None) -> np.ndarray:
    """D = act(alpha * C_ref + beta * C_in + bias) in fp64 for the block of
    C_ref (the same rows/cols lists given to gemm_ref); see gemm_oracle.c."""
    lib = _load()
    C_ref = np.ascontiguousarray(C_ref, dtype=np.float64)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else len(r)
    nc = N if c is None else len(c)
    D = np.zeros((nr, nc), dtype=np.float64)
    if nr == 0 or nc == 0:
        return D
    cin = None if C_in is None else np.ascontiguousarray(C_in)
    b = None if bias is None else np.ascontiguousarray(bias)
    rc = lib.oracle_epilogue(M, N, C_ref.ctypes.data,
                             None if r is None else r.ctypes.data, nr,
                             None if c is None else c.ctypes.data, nc,
                             float(alpha), float(beta), _ptr(cin), ldc, c_major,
                             DTYPES[c_dtype], _ptr(b), ACTIVATIONS[act], D.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_epilogue rejected the arguments (status {rc})")
    return D


def softmax_ref(M: int, N: int, x: np.ndarray, ldx: int) -> np.ndarray:
    """Row softmax of an fp32 M x N matrix (row pitch ldx) in fp64 (M x N)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.zeros((M, N), dtype=np.float64)
    if M == 0 or N == 0:
        return y
    rc = lib.oracle_softmax_rows(M, N, x.ctypes.data, ldx, y.ctypes.data, N)
    if rc != 0:
        raise ValueError(f"oracle_softmax_rows rejected the arguments (status {rc})")
    return y
