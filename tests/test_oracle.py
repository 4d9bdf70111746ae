"""Pins for the CPU oracle (CPU only).

The oracle is the plain definition C[m,n] = sum_k A(m,k) B(n,k) (fp64) and
S[m,n] = sum_k |A(m,k) B(n,k)| -- the product the CuTe DSL Ampere SGEMM
example checks with einsum("mk,nk->mn") in run(), and the CK Tile practice
GEMM checks with its CPU reference ("Result Verification"). The pages print no
GEMM output values, so the oracle is pinned to things other than itself:

* exact rational brute force (``fractions``) on tiny shapes, every major,
  padded leading dimensions and all three element types, with operands
  decoded by numpy (not by the oracle's decoders);
* the oracle's element decoders against numpy on every f16/bf16 bit pattern
  and on random and special f32 patterns;
* closed forms: all-ones (C = S = K) and the ramp A(m,k) = m+k,
  B(n,k) = n-k (C = K m n + (n-m) K(K-1)/2 - (K-1)K(2K-1)/6);
* identity and permutation operands reproduce / permute the other operand;
* linearity in A on integer data (exact), the transpose identity
  C(B, A) = C(A, B)^T, and layout invariance (the same logical matrices in
  every major and leading dimension give the same bytes);
* sampled rows/columns equal the same rows/columns of the full product;
* float64 numpy matmul (a library routine) agrees within fp64 rounding;
* hand-worked small examples in tests/golden/.

``test_pins_catch_planted_mistakes`` plants plausible mistakes (a dropped
term, a wrong sign, a transposed operand, a wrong leading dimension, a
swapped major) in a wrapper around the oracle, on the CPU, and checks that
each one fails at least one pin.
"""

from __future__ import annotations

import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import datagen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers --

def np_decode(storage: np.ndarray, dtype: str) -> np.ndarray:
    """float64 values of a storage array, decoded by numpy."""
    if dtype == "f32":
        return storage.astype(np.float64)
    if dtype == "f16":
        return storage.view(np.float16).astype(np.float64)
    return (storage.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def logical_from_storage(st, rows, kdim, major, ld, dtype):
    vals = np_decode(st, dtype)
    out = np.empty((rows, kdim), dtype=np.float64)
    for r in range(rows):
        for k in range(kdim):
            out[r, k] = vals[r * ld + k] if major == 0 else vals[k * ld + r]
    return out


def make_case(M, N, K, a_major, b_major, dtype, dist="normal", seed=0,
              lda_pad=0, ldb_pad=0, lo=-5, hi=5):
    lda = (K if a_major == 0 else M) + lda_pad
    ldb = (K if b_major == 0 else N) + ldb_pad
    A = datagen.operand(M, K, major=a_major, ld=lda, dtype=dtype, dist=dist,
                        seed=seed, stream=0, lo=lo, hi=hi)
    B = datagen.operand(N, K, major=b_major, ld=ldb, dtype=dtype, dist=dist,
                        seed=seed, stream=1, lo=lo, hi=hi)
    return A, lda, B, ldb


def run_pins(gemm):
    """Run every structural pin against ``gemm`` (signature of
    oracle.gemm_ref). Returns the list of pins that failed."""
    failed = []

    def check(name, cond):
        if not cond:
            failed.append(name)

    # exact brute force on tiny shapes (normal data: rounding matters)
    for (M, N, K), a_major, b_major, dtype in itertools.product(
            [(1, 1, 1), (2, 3, 4), (3, 2, 5), (4, 4, 3)], (0, 1), (0, 1),
            ("f32", "f16", "bf16")):
        A, lda, B, ldb = make_case(M, N, K, a_major, b_major, dtype, seed=M * 7 + K,
                                   lda_pad=1, ldb_pad=2)
        LA = logical_from_storage(A, M, K, a_major, lda, dtype)
        LB = logical_from_storage(B, N, K, b_major, ldb, dtype)
        C, S = gemm(M, N, K, A, lda, a_major, dtype, B, ldb, b_major, dtype)
        if not (np.all(np.isfinite(C)) and np.all(np.isfinite(S))):
            check(f"brute{(M, N, K, a_major, b_major, dtype)}", False)
            continue
        ok = True
        for m in range(M):
            for n in range(N):
                ex = sum((Fraction(float(LA[m, k])) * Fraction(float(LB[n, k]))
                          for k in range(K)), Fraction(0))
                ab = sum((abs(Fraction(float(LA[m, k])) * Fraction(float(LB[n, k])))
                          for k in range(K)), Fraction(0))
                tol = Fraction(K) * Fraction(2) ** -52 * ab
                ok &= abs(Fraction(float(C[m, n])) - ex) <= tol
                ok &= abs(Fraction(float(S[m, n])) - ab) <= tol
        check(f"brute{(M, N, K, a_major, b_major, dtype)}", ok)

    # integer brute force is exact
    for a_major, b_major in itertools.product((0, 1), (0, 1)):
        M, N, K = 3, 4, 6
        A, lda, B, ldb = make_case(M, N, K, a_major, b_major, "f16", dist="int",
                                   seed=11, lda_pad=3)
        LA = logical_from_storage(A, M, K, a_major, lda, "f16")
        LB = logical_from_storage(B, N, K, b_major, ldb, "f16")
        C, _ = gemm(M, N, K, A, lda, a_major, "f16", B, ldb, b_major, "f16")
        ex = np.array([[sum(int(LA[m, k]) * int(LB[n, k]) for k in range(K))
                        for n in range(N)] for m in range(M)], dtype=np.float64)
        check(f"int-brute{(a_major, b_major)}", np.array_equal(C, ex))

    # all ones: C = S = K
    for K in (1, 7, 64):
        A = np.ones(3 * K, np.float32)
        B = np.ones(2 * K, np.float32)
        C, S = gemm(3, 2, K, A, K, 0, "f32", B, K, 0, "f32")
        check(f"ones{K}", np.all(C == K) and np.all(S == K))

    # ramp closed form
    for M, N, K in ((4, 5, 6), (9, 3, 17)):
        A = np.array([[m + k for k in range(K)] for m in range(M)], np.float32).ravel()
        B = np.array([[n - k for k in range(K)] for n in range(N)], np.float32).ravel()
        C, _ = gemm(M, N, K, A, K, 0, "f32", B, K, 0, "f32")
        m, n = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        closed = K * m * n + (n - m) * K * (K - 1) // 2 - (K - 1) * K * (2 * K - 1) // 6
        check(f"ramp{(M, N, K)}", np.array_equal(C, closed.astype(np.float64)))

    # identity operands, in both majors
    for major in (0, 1):
        M, N = 5, 4
        eye = np.eye(M, dtype=np.float32)                      # A = I (K = M)
        Bl = datagen.logical(N, M, dist="int", seed=3)          # N x K logical
        B = Bl.ravel() if major == 0 else Bl.T.copy().ravel()
        C, _ = gemm(M, N, M, eye.ravel(), M, 0, "f32", B, M if major == 0 else N, major, "f32")
        check(f"identity-A{major}", np.array_equal(C, Bl.T.astype(np.float64)))
        Al = datagen.logical(M, N, dist="int", seed=4)          # B = I (K = N)
        A = Al.ravel() if major == 0 else Al.T.copy().ravel()
        C, _ = gemm(M, N, N, A, N if major == 0 else M, major, "f32",
                    np.eye(N, dtype=np.float32).ravel(), N, 0, "f32")
        check(f"identity-B{major}", np.array_equal(C, Al.astype(np.float64)))

    # permutation: A = P (row m has its one at column pi(m)) -> C[m,n] = B(n, pi(m))
    rng = np.random.default_rng(5)
    pi = rng.permutation(6)
    P = np.zeros((6, 6), np.float32)
    P[np.arange(6), pi] = 1
    Bl = datagen.logical(4, 6, dist="int", seed=6)
    C, _ = gemm(6, 4, 6, P.ravel(), 6, 0, "f32", Bl.ravel(), 6, 0, "f32")
    check("permutation", np.array_equal(C, Bl[:, pi].T.astype(np.float64)))

    # linearity in A (integer data: exact)
    M, N, K = 5, 6, 9
    A1 = datagen.logical(M, K, dist="int", seed=8)
    A2 = datagen.logical(M, K, dist="int", seed=9)
    Bl = datagen.logical(N, K, dist="int", seed=10)
    C1, _ = gemm(M, N, K, A1.ravel(), K, 0, "f32", Bl.ravel(), K, 0, "f32")
    C2, _ = gemm(M, N, K, A2.ravel(), K, 0, "f32", Bl.ravel(), K, 0, "f32")
    C12, _ = gemm(M, N, K, (A1 + A2).ravel(), K, 0, "f32", Bl.ravel(), K, 0, "f32")
    check("linearity", np.array_equal(C12, C1 + C2))

    # transpose: C(N,M; B, A) == C(M,N; A, B)^T, and layout invariance
    M, N, K = 7, 5, 11
    ref = None
    for a_major, b_major in itertools.product((0, 1), (0, 1)):
        A, lda, B, ldb = make_case(M, N, K, a_major, b_major, "bf16", seed=12,
                                   lda_pad=a_major * 3, ldb_pad=b_major)
        C, S = gemm(M, N, K, A, lda, a_major, "bf16", B, ldb, b_major, "bf16")
        Ct, St = gemm(N, M, K, B, ldb, b_major, "bf16", A, lda, a_major, "bf16")
        check(f"transpose{(a_major, b_major)}", np.array_equal(C, Ct.T) and np.array_equal(S, St.T))
        if ref is None:
            ref = C
        check(f"layout{(a_major, b_major)}", np.array_equal(C, ref))

    # sampled rows / columns equal the full product
    M, N, K = 13, 11, 9
    A, lda, B, ldb = make_case(M, N, K, 1, 0, "f32", seed=13)
    Cf, Sf = gemm(M, N, K, A, lda, 1, "f32", B, ldb, 0, "f32")
    rows, cols = np.array([0, 5, 12]), np.array([10, 3])
    Cr, Sr = gemm(M, N, K, A, lda, 1, "f32", B, ldb, 0, "f32", rows=rows)
    Cc, _ = gemm(M, N, K, A, lda, 1, "f32", B, ldb, 0, "f32", cols=cols)
    Cb, _ = gemm(M, N, K, A, lda, 1, "f32", B, ldb, 0, "f32", rows=rows, cols=cols)
    check("sampled", np.array_equal(Cr, Cf[rows]) and np.array_equal(Sr, Sf[rows])
          and np.array_equal(Cc, Cf[:, cols]) and np.array_equal(Cb, Cf[np.ix_(rows, cols)]))

    # numpy float64 matmul (library routine) within fp64 rounding
    M, N, K = 33, 17, 70
    A, lda, B, ldb = make_case(M, N, K, 0, 1, "f32", dist="pm1", seed=14)
    C, S = gemm(M, N, K, A, lda, 0, "f32", B, ldb, 1, "f32")
    LA = A.reshape(M, K).astype(np.float64)
    LB = B.reshape(K, N).T.astype(np.float64)
    check("numpy", np.all(np.abs(C - LA @ LB.T) <= K * 2.0 ** -52 * S)
          and np.allclose(S, np.abs(LA) @ np.abs(LB).T, rtol=1e-14, atol=0))
    return failed


# ------------------------------------------------------------------- tests --

def test_oracle_passes_every_pin():
    assert run_pins(oracle.gemm_ref) == []


def test_decoders_every_16bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        f16 = bits.view(np.float16).astype(np.float64)
        bf16 = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    for i in range(1 << 16):
        got16 = oracle.decode(i, "f16")
        gotbf = oracle.decode(i, "bf16")
        assert (got16 == f16[i]) or (np.isnan(got16) and np.isnan(f16[i])), hex(i)
        assert (gotbf == bf16[i]) or (np.isnan(gotbf) and np.isnan(bf16[i])), hex(i)


def test_decoder_f32_patterns():
    rng = np.random.default_rng(0)
    pats = np.concatenate([rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32),
                           np.array([0, 1, 0x007FFFFF, 0x00800000, 0x3F800000, 0x7F7FFFFF,
                                     0x7F800000, 0x80000001, 0xFF800000], np.uint32)])
    with np.errstate(invalid="ignore"):
        ref = pats.view(np.float32).astype(np.float64)
    for p, r in zip(pats, ref):
        got = oracle.decode(int(p), "f32")
        assert got == r or (np.isnan(got) and np.isnan(r)), hex(int(p))


def test_golden_examples():
    """Hand-worked products (values derived by hand in the fixture file)."""
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    assert cases
    for case in cases:
        M, N, K = case["M"], case["N"], case["K"]
        dt = case["dtype"]
        A = datagen.to_storage(np.array(case["A"], np.float64).ravel(), dt)
        B = datagen.to_storage(np.array(case["B"], np.float64).ravel(), dt)
        C, S = oracle.gemm_ref(M, N, K, A, K, 0, dt, B, K, 0, dt)
        assert np.array_equal(C, np.array(case["C"], np.float64)), case["name"]
        assert np.array_equal(S, np.array(case["S"], np.float64)), case["name"]


def test_integer_workloads_are_exact_in_fp32():
    """The integer configurations keep |C| below 2**24 (so float32(C_ref) is
    exact, whatever the summation order): |C| <= K * max|a| * max|b|."""
    assert 256 * 5 * 5 < 2 ** 24          # 1024 x 512 x 256, values in [-5, 5]
    assert 1037 * 3 * 3 < 2 ** 24         # 4095 x 3071 x 1037, values in [-3, 3]
    assert 8192 * 3 * 3 < 2 ** 24         # 16384 x 256 x 8192, values in [-3, 3]
    A, lda, B, ldb = make_case(40, 30, 256, 0, 0, "f16", dist="int", seed=1025)
    C, _ = oracle.gemm_ref(40, 30, 256, A, lda, 0, "f16", B, ldb, 0, "f16")
    assert np.array_equal(C, np.floor(C)) and np.abs(C).max() <= 256 * 25


def test_rejects_bad_arguments():
    A = np.ones(4, np.float32)
    with pytest.raises(ValueError):
        oracle.gemm_ref(2, 2, 2, A, 1, 0, "f32", A, 2, 0, "f32")   # lda < K
    with pytest.raises(ValueError):
        oracle.gemm_ref(2, 2, 2, A, 2, 0, "f32", A, 2, 0, "f32", rows=[2])
    C, S = oracle.gemm_ref(0, 3, 2, A, 2, 0, "f32", A, 2, 0, "f32")
    assert C.shape == (0, 3)
    C, S = oracle.gemm_ref(2, 2, 0, None, 1, 0, "f32", None, 1, 0, "f32")
    assert np.all(C == 0) and np.all(S == 0)


# ------------------------------------------------- planted-mistake checks --

def _mutant(kind):
    """A plausible mistake, planted in a wrapper around the oracle."""
    def g(M, N, K, A, lda, a_major, a_dt, B, ldb, b_major, b_dt, rows=None, cols=None, **kw):
        if kind == "drop_last_k" and K > 0:
            return oracle.gemm_ref(M, N, K - 1, A, lda, a_major, a_dt, B, ldb, b_major,
                                   b_dt, rows=rows, cols=cols, **kw)
        if kind == "wrong_sign":
            C, S = oracle.gemm_ref(M, N, K, A, lda, a_major, a_dt, B, ldb, b_major, b_dt,
                                   rows=rows, cols=cols, **kw)
            return -C, S
        if kind == "swap_a_major" and M == K:
            return oracle.gemm_ref(M, N, K, A, lda, 1 - a_major, a_dt, B, ldb, b_major,
                                   b_dt, rows=rows, cols=cols, **kw)
        if kind == "transposed_result" and M == N:
            C, S = oracle.gemm_ref(M, N, K, A, lda, a_major, a_dt, B, ldb, b_major, b_dt,
                                   rows=rows, cols=cols, **kw)
            return C.T, S.T
        if kind == "ld_ignored":
            inner_a = K if a_major == 0 else M
            inner_b = K if b_major == 0 else N
            if lda != inner_a or ldb != inner_b:
                # a kernel that assumes packed storage reads the padded buffer
                return oracle.gemm_ref(M, N, K, A, inner_a, a_major, a_dt, B, inner_b,
                                       b_major, b_dt, rows=rows, cols=cols, **kw)
        if kind == "first_term_twice" and K > 1:
            C, S = oracle.gemm_ref(M, N, K, A, lda, a_major, a_dt, B, ldb, b_major, b_dt,
                                   rows=rows, cols=cols, **kw)
            C1, _ = oracle.gemm_ref(M, N, 1, A, lda, a_major, a_dt, B, ldb, b_major, b_dt,
                                    rows=rows, cols=cols, **kw)
            return C + C1, S
        if kind == "no_abs_in_s":
            C, S = oracle.gemm_ref(M, N, K, A, lda, a_major, a_dt, B, ldb, b_major, b_dt,
                                   rows=rows, cols=cols, **kw)
            return C, C.copy()
        return oracle.gemm_ref(M, N, K, A, lda, a_major, a_dt, B, ldb, b_major, b_dt,
                               rows=rows, cols=cols, **kw)
    return g


@pytest.mark.parametrize("kind", ["drop_last_k", "wrong_sign", "swap_a_major",
                                  "transposed_result", "ld_ignored", "first_term_twice",
                                  "no_abs_in_s"])
def test_pins_catch_planted_mistakes(kind):
    with np.errstate(all="ignore"):
        assert run_pins(_mutant(kind)), f"no pin caught the planted mistake {kind!r}"


# ------------------------------------------------------ fused epilogue --
# D = act(alpha * C + beta * C_in + bias): the CuTe Ampere SGEMM example's
# epilogue_op hook with scaling, bias and activation written out.

def epilogue_pins(epi):
    """Every epilogue pin, against the callable `epi` (the oracle's signature);
    raises AssertionError on the first that fails."""
    rng = np.random.default_rng(3)
    M, N = 5, 7
    C = rng.integers(-50, 50, (M, N)).astype(np.float64)
    # identity
    assert np.array_equal(epi(M, N, C, 1.0, 0.0), C)
    # scaling only
    assert np.array_equal(epi(M, N, C, -0.5, 0.0), -0.5 * C)
    # bias broadcast along rows, indexed by the column
    bias = np.arange(N, dtype=np.float32) * 3 - 4
    D = epi(M, N, C, 1.0, 0.0, bias=bias)
    assert np.array_equal(D - C, np.broadcast_to(bias.astype(np.float64), (M, N)))
    # beta * C_in in both layouts of C (and 16-bit storage), dyadic => exact
    Lc = rng.integers(-8, 8, (M, N)).astype(np.float64)
    row_major = np.full(M * (N + 2), np.nan, np.float32).reshape(M, N + 2)
    row_major[:, :N] = Lc
    col_major = np.full(N * (M + 1), np.nan, np.float32).reshape(N, M + 1)
    col_major[:, :M] = Lc.T
    D1 = epi(M, N, C, 1.0, 0.25, C_in=row_major.ravel(), ldc=N + 2, c_major=1)
    D0 = epi(M, N, C, 1.0, 0.25, C_in=col_major.ravel(), ldc=M + 1, c_major=0)
    assert np.array_equal(D1, C + 0.25 * Lc) and np.array_equal(D0, D1)
    bf = datagen.to_storage(Lc.ravel(), "bf16")
    D2 = epi(M, N, C, 1.0, 0.25, C_in=bf, ldc=N, c_major=1, c_dtype="bf16")
    assert np.array_equal(D2, D1)
    # beta == 0 never reads C_in (NaN storage must not leak in)
    nan_c = np.full(M * N, np.nan, np.float32)
    assert np.array_equal(epi(M, N, C, 1.0, 0.0, C_in=nan_c, ldc=N), C)
    # ReLU
    assert np.array_equal(epi(M, N, C, 1.0, 0.0, act="relu"), np.maximum(C, 0))
    # GELU: x * Phi(x); Phi(1) = 0.8413447460685429 (normal table), odd part = x
    g = epi(1, 5, np.array([[1.0, -1.0, 0.0, 10.0, -10.0]]), 1.0, 0.0,
                            act="gelu")[0]
    assert abs(g[0] - 0.8413447460685429) < 1e-15
    assert abs(g[1] + (1 - 0.8413447460685429)) < 1e-15
    assert g[2] == 0.0 and abs(g[3] - 10.0) < 1e-15 and abs(g[4]) < 1e-15
    assert abs((g[0] - g[1]) - 1.0) < 1e-15
    # sampled block equals the same block of the full result
    rows, cols = np.array([4, 0]), np.array([6, 2, 3])
    Db = epi(M, N, C[np.ix_(rows, cols)], 2.0, 0.25, C_in=row_major.ravel(),
                             ldc=N + 2, c_major=1, bias=bias, act="relu", rows=rows, cols=cols)
    Df = epi(M, N, C, 2.0, 0.25, C_in=row_major.ravel(), ldc=N + 2,
                             c_major=1, bias=bias, act="relu")
    assert np.array_equal(Db, Df[np.ix_(rows, cols)])


def test_epilogue_pins():
    epilogue_pins(oracle.epilogue_ref)


def test_epilogue_rejects_bad_arguments():
    C = np.zeros((2, 2))
    with pytest.raises(ValueError):
        oracle.epilogue_ref(2, 2, C, 1.0, 0.5)              # beta != 0 without C_in
    with pytest.raises(ValueError):
        oracle.epilogue_ref(2, 2, C, 1.0, 0.0, rows=[2])    # row out of range


# ------------------------------------------------------------ row softmax --
# The Gluon Multi-CTA tutorial's multi-CTA softmax: y = exp(x - max) / sum.

def softmax_pins(smx):
    """Every softmax pin, against the callable `smx` (the oracle's
    signature); raises AssertionError on the first that fails."""
    import math
    # hand-worked: x = [0, ln 2, ln 5] -> [1, 2, 5] / 8
    x = np.array([0.0, math.log(2.0), math.log(5.0)], np.float32)
    y = smx(1, 3, x, 3)[0]
    xd = x.astype(np.float64)
    want = np.exp(xd - xd.max()) / np.exp(xd - xd.max()).sum()
    assert np.allclose(y, want, rtol=1e-15, atol=0)
    assert abs(y[0] - 1 / 8) < 1e-7 and abs(y[2] - 5 / 8) < 1e-7
    # uniform rows give 1/N; rows sum to one; shift invariance; padding ignored
    rng = np.random.default_rng(4)
    M, N, ld = 6, 37, 40
    xs = np.full(M * ld, np.nan, np.float32)
    body = (rng.integers(-64, 64, (M, N)) / 8.0).astype(np.float32)  # exact under +16
    xs.reshape(M, ld)[:, :N] = body
    y = smx(M, N, xs, ld)
    assert np.allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    shifted = xs.copy()
    shifted.reshape(M, ld)[:, :N] += 16.0
    assert np.array_equal(shifted.reshape(M, ld)[:, :N] - 16.0, body)
    assert np.allclose(smx(M, N, shifted, ld), y, rtol=1e-13, atol=0)
    assert np.allclose(smx(2, 9, np.full(18, 1.5, np.float32), 9), 1 / 9,
                       rtol=1e-15, atol=0)
    # monotone in x, and the largest input gets the largest output
    assert all(np.argmax(y[i]) == np.argmax(body[i]) for i in range(M))
    order = np.argsort(body[0])
    assert np.all(np.diff(y[0][order]) >= 0)
    # a dominant entry takes (almost) all the mass
    xd = np.zeros(50, np.float32)
    xd[7] = 60.0
    yd = smx(1, 50, xd, 50)[0]
    assert abs(yd[7] - 1.0) < 1e-24 and yd[0] == np.exp(-60.0) * yd[7]
    # a large-magnitude row: without the max shift exp() overflows even in fp64
    big = np.array([-5.0, 800.0, 3.0, 800.0], np.float32)
    yb = smx(1, 4, big, 4)[0]
    assert np.all(np.isfinite(yb)) and yb[1] == 0.5 and yb[3] == 0.5 and yb[0] == 0.0


def test_softmax_pins():
    softmax_pins(oracle.softmax_ref)


# ---------------------------- planted mistakes in the epilogue and softmax --

def _epilogue_mutant(kind):
    """A plausible epilogue mistake, planted in a wrapper around the oracle."""
    import math

    def g(M, N, C_ref, alpha, beta, C_in=None, ldc=0, c_major=1, c_dtype="f32", bias=None,
          act="none", rows=None, cols=None):
        kw = dict(C_in=C_in, ldc=ldc, c_major=c_major, c_dtype=c_dtype, rows=rows, cols=cols)
        if kind == "alpha_ignored":
            return oracle.epilogue_ref(M, N, C_ref, 1.0, beta, bias=bias, act=act, **kw)
        if kind == "beta_ignored":
            return oracle.epilogue_ref(M, N, C_ref, alpha, 0.0, bias=bias, act=act, **kw)
        if kind == "c_in_layout_swapped" and C_in is not None:
            kw["c_major"] = 1 - c_major
            return oracle.epilogue_ref(M, N, C_ref, alpha, beta, bias=bias, act=act, **kw)
        if kind == "bias_by_row" and bias is not None and act == "none":
            D = oracle.epilogue_ref(M, N, C_ref, alpha, beta, act=act, **kw)
            r = np.arange(M) if rows is None else np.asarray(rows)
            return D + np.asarray(bias, np.float64)[r % len(bias)][:, None]
        if kind == "gelu_without_half" and act == "gelu":
            pre = oracle.epilogue_ref(M, N, C_ref, alpha, beta, bias=bias, act="none", **kw)
            return pre * (1.0 + np.vectorize(math.erf)(pre / math.sqrt(2.0)))
        if kind == "relu_as_abs" and act == "relu":
            pre = oracle.epilogue_ref(M, N, C_ref, alpha, beta, bias=bias, act="none", **kw)
            return np.abs(pre)
        return oracle.epilogue_ref(M, N, C_ref, alpha, beta, bias=bias, act=act, **kw)
    return g


@pytest.mark.parametrize("kind", ["alpha_ignored", "beta_ignored", "c_in_layout_swapped",
                                  "bias_by_row", "gelu_without_half", "relu_as_abs"])
def test_epilogue_pins_catch_planted_mistakes(kind):
    with np.errstate(all="ignore"), pytest.raises(AssertionError):
        epilogue_pins(_epilogue_mutant(kind))


def _softmax_mutant(kind):
    """A plausible softmax mistake, planted in a wrapper around the oracle."""
    def rows_of(M, N, x, ldx):
        x = np.asarray(x, np.float32)
        return np.stack([x[m * ldx:m * ldx + N].astype(np.float64) for m in range(M)])

    def g(M, N, x, ldx):
        if kind == "no_max_shift":
            e = np.exp(rows_of(M, N, x, ldx))
            return e / e.sum(axis=1, keepdims=True)
        if kind == "shift_by_first_value":
            r = rows_of(M, N, x, ldx)
            e = np.exp(r - r[:, :1])
            return e / e.sum(axis=1, keepdims=True)
        if kind == "not_normalised":
            r = rows_of(M, N, x, ldx)
            return np.exp(r - r.max(axis=1, keepdims=True))
        if kind == "ld_ignored" and ldx != N:
            return oracle.softmax_ref(M, N, x, N)
        if kind == "last_column_dropped" and N > 1:
            y = np.zeros((M, N))
            xs = np.asarray(x, np.float32)
            packed = np.concatenate([xs[m * ldx:m * ldx + N - 1] for m in range(M)])
            y[:, :N - 1] = oracle.softmax_ref(M, N - 1, packed, N - 1)
            return y
        return oracle.softmax_ref(M, N, x, ldx)
    return g


@pytest.mark.parametrize("kind", ["no_max_shift", "shift_by_first_value", "not_normalised",
                                  "ld_ignored", "last_column_dropped"])
def test_softmax_pins_catch_planted_mistakes(kind):
    with np.errstate(all="ignore"), pytest.raises(AssertionError):
        softmax_pins(_softmax_mutant(kind))
