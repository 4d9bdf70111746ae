"""The acceptance rules themselves (CPU only)."""

import numpy as np

from acceptance import assert_accepted, exact_integer_case, ulp, violations


def test_ulp_matches_numpy_spacing():
    rng = np.random.default_rng(1)
    x16 = np.concatenate([rng.normal(0, 100, 2000), [1.0, 2.0, 6.1e-5, 1e-7]])
    ref16 = np.spacing(np.abs(x16.astype(np.float16))).astype(np.float64)
    assert np.array_equal(ulp(x16.astype(np.float16).astype(np.float64), "f16"), ref16)
    assert ulp(np.array([65504.0]), "f16")[0] == 32.0  # numpy's spacing overflows there
    x32 = np.concatenate([rng.normal(0, 1e3, 2000), [1.0, 1e-40, 3.0e38]])
    ref32 = np.spacing(np.abs(x32.astype(np.float32))).astype(np.float64)
    assert np.array_equal(ulp(x32.astype(np.float32).astype(np.float64), "f32"), ref32)


def test_ulp_bf16_by_bit_stepping():
    for v in [1.0, 1.5, 3.0, 255.0, 1e-3, -7.25, 1e30]:
        b = (np.array([v], np.float32).view(np.uint32) >> 16).astype(np.uint32)
        lo = (b << 16).view(np.float32)[0]
        hi = ((b + 1) << 16).view(np.float32)[0]
        assert ulp(np.array([lo], np.float64), "bf16")[0] == abs(float(hi) - float(lo))
    assert ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7
    assert ulp(np.array([0.0]), "bf16")[0] == 2.0 ** -133


def test_rules():
    C_ref = np.array([1.0, 100.0, 0.0, 3.0])
    S = np.array([10.0, 1000.0, 0.0, 3.0])
    ok = C_ref + np.array([9e-4, 0.09, 0.0, 0.0])
    assert not violations(ok, C_ref, S, "f32")[0].any()
    bad = C_ref + np.array([2e-3, 0.0, 0.0, 0.0])
    assert violations(bad, C_ref, S, "f32")[0].tolist() == [True, False, False, False]
    # S == 0 demands an exact zero; NaN always fails
    assert violations(np.array([1.0, 100.0, 1e-30, np.nan]), C_ref, S, "bf16")[0].tolist() == \
        [False, False, True, True]
    # 16-bit outputs get one ulp on top of the relative term
    assert not violations(np.array([100.5]), np.array([100.0]), np.array([0.0001]), "bf16")[0].any()
    # exact rule compares with float32(C_ref)
    assert violations(np.array([3.0, 4.0]), np.array([3.0, 4.0]), S[:2], "f32", exact=True)[0].sum() == 0
    assert violations(np.array([3.0, 4.5]), np.array([3.0, 4.0]), S[:2], "f32", exact=True)[0].sum() == 1
    assert exact_integer_case(np.array([1.0, -6400.0])) and not exact_integer_case(np.array([0.5]))
    assert_accepted(ok, C_ref, S, "f32", what="sanity")
