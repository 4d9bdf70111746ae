"""Acceptance rules for a GEMM result against the oracle (test infrastructure).

Rules (the contract for this library; the pages themselves compare against a
library product with fixed atol/rtol -- the CuTe Ampere SGEMM example with
atol 1e-3 / rtol 1e-5, the Gluon Multi-CTA tutorial with atol 0.1 / rtol
0.01 -- which we replace by a per-element bound that scales with the sum):

* integer-valued inputs whose partial sums stay below 2**24: bit-exact,
  ``C == float32(C_ref)`` (every partial sum is an exactly representable
  integer in fp32 whatever the summation order, and the 16-bit products are
  exact in the tensor cores' fp32 accumulation);
* fp32 output: ``|C - C_ref| <= 1e-4 * S`` with ``S = sum_k |a_k b_k|``;
* bf16/fp16 output: ``|C - C_ref| <= ulp_out(C_ref) + 1e-4 * S``, where
  ``ulp_out(x)`` is the spacing of the output type at ``|x|``:
  ``2**(floor(log2|x|) - p + 1)`` with ``p`` the type's significand bits
  (24 f32, 11 f16, 8 bf16), and the subnormal spacing below the smallest
  normal;
* where ``S == 0`` the result must be exactly zero; a NaN anywhere fails.
"""

from __future__ import annotations

import numpy as np

PRECISION = {"f32": (24, -126), "f16": (11, -14), "bf16": (8, -126)}
REL = 1e-4


def ulp(x, dtype: str) -> np.ndarray:
    """Spacing of ``dtype`` at ``|x|`` (float64 array)."""
    p, emin = PRECISION[dtype]
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(ax > 0, ax, 1.0))  # ax = f * 2**e, f in [0.5, 1)
    e = np.maximum(e - 1, emin)                  # floor(log2 ax), clamped to normals
    e = np.where(ax > 0, e, emin)
    return np.ldexp(1.0, (e - (p - 1)).astype(np.int64))


def bound(C_ref, S, out_dtype: str) -> np.ndarray:
    b = REL * np.asarray(S, dtype=np.float64)
    if out_dtype != "f32":
        b = b + ulp(C_ref, out_dtype)
    return b


def violations(C, C_ref, S, out_dtype: str, exact: bool = False):
    """Boolean mask of elements that break the rule, and the worst ratio."""
    C = np.asarray(C, dtype=np.float64)
    C_ref = np.asarray(C_ref, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    bad = ~np.isfinite(C)
    if exact:
        bad |= C != C_ref.astype(np.float32).astype(np.float64)
        return bad, float(bad.any())
    err = np.abs(C - C_ref)
    lim = bound(C_ref, S, out_dtype)
    bad |= err > lim
    bad |= (S == 0) & (C != 0)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(lim > 0, err / lim, np.where(err > 0, np.inf, 0.0))
    return bad, float(np.nanmax(ratio)) if ratio.size else 0.0


def assert_accepted(C, C_ref, S, out_dtype: str, exact: bool = False, what: str = ""):
    bad, worst = violations(C, C_ref, S, out_dtype, exact)
    if bad.any():
        idx = np.argwhere(bad)
        first = tuple(int(i) for i in idx[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside the rule "
            f"(exact={exact}); first at {first}: got {np.asarray(C)[first]!r}, "
            f"oracle {np.asarray(C_ref)[first]!r}, S {np.asarray(S)[first]!r}; "
            f"worst err/bound {worst:.3g}")
    return worst


def exact_integer_case(C_ref) -> bool:
    """True when every C_ref is an integer of magnitude below 2**24."""
    C_ref = np.asarray(C_ref)
    return bool(np.all(np.floor(C_ref) == C_ref) and np.all(np.abs(C_ref) < 2 ** 24))
