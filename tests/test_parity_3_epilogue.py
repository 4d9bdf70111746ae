"""GPU parity of gemm_ex: C = act(alpha * A B^T + beta * C + bias[n]), the
fused epilogue (the CuTe Ampere SGEMM example's epilogue_op hook) on both
kernel families, every type, both C layouts and three activations, against
the oracle's epilogue applied to its fp64 product.

Integer inputs with dyadic alpha/beta keep every intermediate exact in fp32,
so identity and ReLU results are compared bit-exactly (16-bit outputs with
round-to-nearest-even of the exact value). GELU goes through erff and is
compared within 1.2e-4 * S_epi + 1e-6 * (|D_ref| + 1) (+1 output ulp), where
S_epi = |alpha| S + |beta C_old| + |bias| bounds the pre-activation's
rounding and GELU's slope is below 1.13."""

import itertools

import numpy as np
import pytest

import datagen
import dense_gemm_06_gb300 as lg
import oracle
from acceptance import ulp
from gpu_util import CBuffer, decode, make_operands, to_device

pytestmark = pytest.mark.gpu

ACTS = {"none": lg.GEMM_ACT_NONE, "relu": lg.GEMM_ACT_RELU, "gelu": lg.GEMM_ACT_GELU}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


def rne_out(x, t):
    if t == "f32":
        return x.astype(np.float32).astype(np.float64)
    if t == "f16":
        return x.astype(np.float16).astype(np.float64)
    bits = datagen.f32_to_bf16_bits(x.astype(np.float32))
    return decode(bits, "bf16")


def run_ex(M, N, K, dtype, am, bm, cm, act, alpha, beta, with_bias, seed, ldc_pad=0):
    import torch
    it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
    A, lda, B, ldb = make_operands(M, N, K, dtype, am, bm, "int", seed, lo=-3, hi=3)
    ldc = (N if cm == lg.GEMM_MAJOR_MN else M) + ldc_pad
    cbuf = CBuffer(M, N, cm, ldc, ot)
    Lc = datagen.logical(M, N, dtype=ot, dist="int", lo=-4, hi=4, seed=seed, stream=7)
    c_store = cbuf.fill(Lc)
    bias = datagen.logical(1, N, dtype=ot, dist="int", lo=-9, hi=9, seed=seed, stream=8)[0] \
        if with_bias else None
    dbias = to_device(bias) if with_bias else None
    dA, dB = (to_device(A), to_device(B)) if K else (None, None)
    rc = lg.gemm_ex(M, N, K, dA if dA is not None else 0, lda, am,
                    dB if dB is not None else 0, ldb, bm, cbuf.ptr(), ldc, cm, dtype,
                    alpha=alpha, beta=beta, bias=dbias, activation=ACTS[act])
    lg.check(rc, "gemm_ex")
    lg.check(lg.gemm_check_device_error(), "device error word")
    torch.cuda.synchronize()
    D = cbuf.read()
    C_ref, S = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, bm, it)
    D_ref = oracle.epilogue_ref(M, N, C_ref, alpha, beta, C_in=c_store, ldc=ldc, c_major=cm,
                                c_dtype=ot, bias=bias, act=act)
    what = f"{M}x{N}x{K} dtype={dtype} C{'MN'[cm]} act={act} beta={beta} bias={with_bias}"
    if act in ("none", "relu"):
        want = rne_out(D_ref, ot)
        bad = D != want
        assert not bad.any(), f"{what}: {int(bad.sum())} elements differ"
    else:
        s_epi = abs(alpha) * S + abs(beta) * np.abs(decode(Lc, ot)) + \
            (np.abs(decode(bias, ot))[None, :] if with_bias else 0)
        lim = 1.2e-4 * s_epi + 1e-6 * (np.abs(D_ref) + 1)
        if ot != "f32":
            lim = lim + ulp(D_ref, ot)
        err = np.abs(D - D_ref)
        assert np.all(err <= lim), f"{what}: worst err/bound {np.max(err / lim):.3g}"


TYPES = [lg.GEMM_F32, lg.GEMM_F16_F32, lg.GEMM_BF16_F32, lg.GEMM_F16_F16, lg.GEMM_BF16_BF16]


@pytest.mark.parametrize("beta,with_bias", [(0.0, False), (0.25, True)])
@pytest.mark.parametrize("act", sorted(ACTS))
@pytest.mark.parametrize("cm", [0, 1])
@pytest.mark.parametrize("dtype", TYPES)
def test_gemm_ex(dtype, cm, act, beta, with_bias):
    run_ex(300, 520, 200, dtype, 0, 1, cm, act, 0.5, beta, with_bias, seed=21)


@pytest.mark.parametrize("dtype", [lg.GEMM_F32, lg.GEMM_BF16_BF16])
@pytest.mark.parametrize("am,bm", list(itertools.product((0, 1), (0, 1))))
def test_gemm_ex_ragged_and_misaligned(dtype, am, bm):
    # ragged M/N/K and an odd ldc (scalar epilogue path)
    run_ex(257, 131, 77, dtype, am, bm, 1, "relu", -1.5, 0.5, True, seed=22, ldc_pad=1)
    run_ex(129, 263, 1037, dtype, am, bm, 0, "none", 2.0, 0.75, True, seed=23, ldc_pad=3)


@pytest.mark.parametrize("dtype", [lg.GEMM_F32, lg.GEMM_F16_F16])
def test_gemm_ex_k_zero(dtype):
    # no product term: C = act(beta * C + bias)
    run_ex(37, 45, 0, dtype, 0, 0, 1, "relu", 3.0, 0.5, True, seed=24, ldc_pad=3)
    run_ex(37, 45, 0, dtype, 0, 0, 0, "none", 3.0, -1.0, False, seed=25)


def test_gemm_ex_plain_is_gemm():
    # alpha 1, beta 0, no bias, no activation: the plain gemm() path
    run_ex(300, 520, 200, lg.GEMM_BF16_F32, 0, 0, 1, "none", 1.0, 0.0, False, seed=26)


@pytest.mark.parametrize("act", sorted(ACTS))
def test_gemm_ex_with_split_tail(act):
    # the fixup kernel of the FFMA kernel's K-split applies the epilogue
    old = lg.gemm_get_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL)
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 2))
    try:
        run_ex(300, 261, 70, lg.GEMM_F32, 0, 1, 1, act, 0.5, 0.25, True, seed=31, ldc_pad=3)
        run_ex(130, 77, 40, lg.GEMM_F32, 1, 0, 0, act, -1.0, 0.0, False, seed=32)
    finally:
        lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, old)


@pytest.mark.parametrize("act", sorted(ACTS))
def test_gemm_ex_tma_fed_ffma(act):
    # FFMA configuration 9 (TMA-fed, MN-major operands with 16-byte pitches)
    old = lg.gemm_get_option(lg.GEMM_OPT_SIMT_CONFIG)
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, 9))
    try:
        run_ex(300, 520, 200, lg.GEMM_F32, 1, 1, 1, act, 0.5, 0.25, True, seed=33)
        run_ex(132, 260, 77, lg.GEMM_F32, 1, 1, 0, act, -1.0, 0.0, False, seed=34, ldc_pad=3)
    finally:
        lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, old)
