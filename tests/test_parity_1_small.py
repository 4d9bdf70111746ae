"""GPU parity on small and ragged shapes, every type, major and kernel variant.

Shapes span several tiles of both kernels (128 x 128 x 16 FFMA tiles,
128/256 x 256 x 64 tensor-core tiles) and leave ragged tails in M, N and K,
as the CuTe Ampere SGEMM example's predicated tails and the Gluon Multi-CTA
tutorial's partial tiles require. Integer-valued inputs are compared
bit-exactly (fp32 output: C == C_ref; 16-bit output: C == round-to-nearest-
even(C_ref)); float inputs under |C - C_ref| <= 1e-4 * S (+1 ulp)."""

import itertools

import numpy as np
import pytest

import datagen
import dense_gemm_06_gb300 as lg
from gpu_util import check_full, make_operands, run_device_gemm

pytestmark = pytest.mark.gpu

TC_TYPES = [lg.GEMM_F16_F32, lg.GEMM_BF16_F32, lg.GEMM_F16_F16, lg.GEMM_BF16_BF16]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


def rne16(x: np.ndarray, t: str) -> np.ndarray:
    """Round exact (integer-valued) results to the 16-bit output type."""
    if t == "f16":
        return x.astype(np.float16).astype(np.float64)
    bits = datagen.f32_to_bf16_bits(x.astype(np.float32))
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# tensor-core kernel modes: (CTA group, operand multicast across two pairs,
# tile scheduler: 1 static persistent, 2 cluster launch control)
TC_MODES = {"cg1": (1, 1, 1), "cg2": (2, 1, 1), "cg2mc": (2, 2, 1), "cg1clc": (1, 1, 2),
            "cg2clc": (2, 1, 2), "auto": (0, 0, 0)}


def run_and_check(M, N, K, dtype, am, bm, cm=1, dist="int", seed=0, lda_pad=0, ldb_pad=0,
                  ldc_pad=0, cta_group=0, tc_store=0, multicast=0, scheduler=0, tile_n=0,
                  split=0):
    A, lda, B, ldb = make_operands(M, N, K, dtype, am, bm, dist, seed, lda_pad, ldb_pad)
    C = run_device_gemm(M, N, K, dtype, A, lda, am, B, ldb, bm, cm, ldc_pad, cta_group,
                        tc_store=tc_store, multicast=multicast, scheduler=scheduler,
                        tile_n=tile_n, split=split)
    what = (f"{M}x{N}x{K} dtype={dtype} A{'KM'[am]} B{'KN'[bm]} C{'MN'[cm]} cg={cta_group} "
            f"store={tc_store} mc={multicast} sched={scheduler} tile_n={tile_n} split={split}")
    ot = lg.OUT_TYPE[dtype]
    if dist == "int" and ot != "f32":
        import oracle
        it = lg.IN_TYPE[dtype]
        C_ref, _ = oracle.gemm_ref(M, N, K, A, lda, am, it, B, ldb, bm, it, with_s=False)
        want = rne16(C_ref, ot)
        bad = C != want
        assert not bad.any(), f"{what}: {int(bad.sum())} elements differ from RNE(C_ref)"
        return
    check_full(C, M, N, K, dtype, A, lda, am, B, ldb, bm, exact=(dist == "int"), what=what)


# ----------------------------------------------------------- FFMA kernel --

SIMT_SHAPES = [(1, 1, 1), (15, 17, 7), (127, 129, 65), (130, 260, 300), (257, 131, 33)]


@pytest.mark.parametrize("shape", SIMT_SHAPES)
@pytest.mark.parametrize("am,bm,cm", list(itertools.product((0, 1), (0, 1), (0, 1))))
def test_sgemm_ragged(shape, am, bm, cm):
    M, N, K = shape
    run_and_check(M, N, K, lg.GEMM_F32, am, bm, cm, dist="pm1", seed=M + N + K)


@pytest.mark.parametrize("am,bm", list(itertools.product((0, 1), (0, 1))))
def test_sgemm_padded_and_unaligned_ld(am, bm):
    # odd leading dimensions: the MN-major operands take the 4-byte copy path
    run_and_check(200, 150, 90, lg.GEMM_F32, am, bm, 1, dist="int", seed=3,
                  lda_pad=3, ldb_pad=5, ldc_pad=1)
    run_and_check(200, 150, 90, lg.GEMM_F32, am, bm, 0, dist="int", seed=4,
                  lda_pad=4, ldb_pad=8, ldc_pad=4)


# ---------------------------------------------------- tcgen05 kernel --

TC_SHAPES = [(1, 1, 1), (100, 70, 64), (300, 520, 200), (257, 513, 1037)]


@pytest.mark.parametrize("tc_store", [0, 1])
@pytest.mark.parametrize("mode", sorted(TC_MODES))
@pytest.mark.parametrize("dtype", TC_TYPES)
@pytest.mark.parametrize("am,bm", list(itertools.product((0, 1), (0, 1))))
@pytest.mark.parametrize("shape", TC_SHAPES)
def test_tc_ragged_integer(shape, am, bm, dtype, mode, tc_store):
    # tc_store 0: TMA store of C where its rows are 16-byte aligned; 1: st.global
    M, N, K = shape
    cg, mc, sch = TC_MODES[mode]
    run_and_check(M, N, K, dtype, am, bm, 1, dist="int", seed=K, cta_group=cg,
                  tc_store=tc_store, multicast=mc, scheduler=sch)


@pytest.mark.parametrize("tc_store", [0, 1])
@pytest.mark.parametrize("mode", sorted(TC_MODES))
@pytest.mark.parametrize("dtype", TC_TYPES)
@pytest.mark.parametrize("cm", [0, 1])
def test_tc_normal_values(dtype, cm, mode, tc_store):
    cg, mc, sch = TC_MODES[mode]
    run_and_check(384, 520, 640, dtype, 0, 1, cm, dist="normal", seed=5, cta_group=cg,
                  tc_store=tc_store, multicast=mc, scheduler=sch)


@pytest.mark.parametrize("mode", sorted(TC_MODES))
@pytest.mark.parametrize("am,bm", list(itertools.product((0, 1), (0, 1))))
def test_tc_misaligned_leading_dims(am, bm, mode):
    # leading dimensions that are not 16-byte multiples force the repack path;
    # an odd ldc forces predicated scalar stores
    cg, mc, sch = TC_MODES[mode]
    run_and_check(333, 277, 131, lg.GEMM_F16_F32, am, bm, 1, dist="int", seed=6,
                  lda_pad=1, ldb_pad=3, ldc_pad=1, cta_group=cg, multicast=mc, scheduler=sch)
    run_and_check(333, 277, 131, lg.GEMM_BF16_BF16, am, bm, 0, dist="normal", seed=7,
                  lda_pad=5, ldb_pad=1, ldc_pad=3, cta_group=cg, multicast=mc, scheduler=sch)


@pytest.mark.parametrize("mode", sorted(TC_MODES))
def test_tc_many_tiles_per_cta(mode):
    # more tiles than CTA pairs: exercises the TMEM double buffer and the
    # smem ring phases across tiles; an odd number of tile rows (11) leaves
    # the second pair of a multicast cluster without rows on the last units
    cg, mc, sch = TC_MODES[mode]
    run_and_check(2560, 2304, 320, lg.GEMM_F16_F32, 0, 0, 1, dist="int", seed=9,
                  cta_group=cg, multicast=mc, scheduler=sch)
    run_and_check(2816, 1280, 200, lg.GEMM_BF16_F32, 1, 1, 1, dist="int", seed=10,
                  cta_group=cg, multicast=mc, scheduler=sch)


@pytest.mark.parametrize("split", [1, 2])
@pytest.mark.parametrize("sched", [1, 2])
@pytest.mark.parametrize("cg,tile_n", [(1, 64), (1, 128), (1, 256), (2, 128), (2, 256)])
@pytest.mark.parametrize("am,bm", list(itertools.product((0, 1), (0, 1))))
def test_tc_tile_widths_and_split_units(am, bm, cg, tile_n, sched, split):
    # every tile width, with the last round's tiles run whole (split 1) or as
    # two half-width units (split 2; every tile here, under one round), under
    # both tile schedulers; ragged M, N and K
    run_and_check(777, 1000, 333, lg.GEMM_F16_F32, am, bm, 1, dist="int", seed=11,
                  cta_group=cg, scheduler=sched, tile_n=tile_n, split=split)
    run_and_check(333, 650, 130, lg.GEMM_BF16_BF16, am, bm, 0, dist="normal", seed=12,
                  cta_group=cg, scheduler=sched, tile_n=tile_n, split=split)


@pytest.mark.parametrize("cg,tile_n", [(1, 128), (2, 256)])
def test_tc_split_last_round_of_many(cg, tile_n):
    # more tiles than resident clusters: the last round's tiles run as half
    # units after whole tiles (auto and forced), int data compared exactly
    for split in (0, 2):
        run_and_check(4736, 2304, 192, lg.GEMM_F16_F32, 0, 1, 1, dist="int", seed=13,
                      cta_group=cg, tile_n=tile_n, split=split)


@pytest.mark.parametrize("shape", [(1000, 1001, 333), (300, 520, 2000), (2048, 2048, 256),
                                   (129, 257, 17)])
def test_sgemm_stream_k(shape):
    # the TMA-fed FFMA kernel (MN-major operands, 16-byte rows) with stream-K
    # forced: a third of the tiles whole, the others' k-iterations shared by
    # 1.5x as many CTAs (ranges crossing tile boundaries, partial tiles summed
    # in k order by the fixup kernel); integer data, so the sum is exact
    M, N, K = shape
    saved = lg.gemm_get_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL)
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 3))
    try:
        run_and_check(M, N, K, lg.GEMM_F32, 1, 1, 1, dist="int", seed=M + K)
        run_and_check(M, N, K, lg.GEMM_F32, 1, 1, 0, dist="pm1", seed=K)
    finally:
        lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, saved)


# ----------------------------------------------------- degenerate sizes --

@pytest.mark.parametrize("dtype", [lg.GEMM_F32, lg.GEMM_BF16_F32, lg.GEMM_F16_F16])
def test_k_zero_writes_zero(dtype):
    C = run_device_gemm(37, 45, 0, dtype, np.zeros(0, np.float32), 1, 0,
                        np.zeros(0, np.float32), 1, 0, 1, ldc_pad=3)
    assert np.all(C == 0)


@pytest.mark.parametrize("dtype", [lg.GEMM_F32, lg.GEMM_BF16_F32])
def test_empty_m_or_n_is_a_no_op(dtype):
    A, lda, B, ldb = make_operands(5, 6, 7, dtype, 0, 0, "int", 1)
    n0 = lg.gemm_launch_count()
    C = run_device_gemm(0, 6, 7, dtype, A[:0], lda, 0, B, ldb, 0)
    assert C.shape == (0, 6)
    C = run_device_gemm(5, 0, 7, dtype, A, lda, 0, B[:0], ldb, 0)
    assert C.shape == (5, 0)
    assert lg.gemm_launch_count() == n0


@pytest.mark.parametrize("dtype", [lg.GEMM_F32, lg.GEMM_F16_F32])
def test_k_one(dtype):
    run_and_check(129, 257, 1, dtype, 1, 0, 1, dist="int", seed=2)


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5, 6, 7, 8, 9])
@pytest.mark.parametrize("am,bm", list(itertools.product((0, 1), (0, 1))))
def test_sgemm_every_tile_config(config, am, bm):
    old = lg.gemm_get_option(lg.GEMM_OPT_SIMT_CONFIG)
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, config))
    try:
        run_and_check(257, 131, 100, lg.GEMM_F32, am, bm, 1, dist="pm1", seed=config)
        run_and_check(130, 260, 77, lg.GEMM_F32, am, bm, 0, dist="int", seed=config,
                      lda_pad=1, ldb_pad=2)
    finally:
        lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, old)


@pytest.mark.parametrize("transpose", [1, 2])
@pytest.mark.parametrize("am,bm,cm", list(itertools.product((0, 1), (0, 1), (0, 1))))
def test_sgemm_with_and_without_operand_transpose(transpose, am, bm, cm):
    old = lg.gemm_get_option(lg.GEMM_OPT_SIMT_TRANSPOSE)
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_TRANSPOSE, transpose))
    try:
        run_and_check(301, 163, 97, lg.GEMM_F32, am, bm, cm, dist="pm1", seed=11,
                      lda_pad=3, ldb_pad=1, ldc_pad=2)
        run_and_check(64, 96, 33, lg.GEMM_F32, am, bm, cm, dist="int", seed=12)
    finally:
        lg.gemm_set_option(lg.GEMM_OPT_SIMT_TRANSPOSE, old)


# K-split of the FFMA kernel's last wave (GEMM_OPT_SIMT_SPLIT_TAIL): forced on
# small and ragged shapes (every tile split, slices of one k-tile or empty),
# and the automatic rule on a shape whose last wave is nearly empty.
@pytest.mark.parametrize("config", [1, 5, 7, 9])
@pytest.mark.parametrize("am,bm,cm", list(itertools.product((0, 1), (0, 1), (0, 1))))
def test_sgemm_split_tail_forced(config, am, bm, cm):
    old = {o: lg.gemm_get_option(o) for o in (lg.GEMM_OPT_SIMT_SPLIT_TAIL,
                                              lg.GEMM_OPT_SIMT_CONFIG)}
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 2))
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, config))
    try:
        for i, (M, N, K) in enumerate([(1, 1, 1), (15, 17, 7), (130, 260, 300), (257, 131, 33)]):
            run_and_check(M, N, K, lg.GEMM_F32, am, bm, cm, dist="int", seed=40 + i,
                          lda_pad=i % 2, ldc_pad=i % 3)
        run_and_check(300, 520, 200, lg.GEMM_F32, am, bm, cm, dist="pm1", seed=45)
    finally:
        for o, v in old.items():
            lg.gemm_set_option(o, v)


# Configuration 9 fills shared memory with TMA tensor copies when both
# operands are MN-major with 16-byte aligned pitches (the pitch of n fp32
# elements padded to a multiple of 4 here); shapes leave ragged M, N and K
# (K below one 16-deep k-tile, and long enough to wrap the 5-stage ring many
# times), and both C layouts swap which operand is A.
def pad4(n: int) -> int:
    return (-n) % 4


def with_options(opts: dict, fn):
    old = {o: lg.gemm_get_option(o) for o in opts}
    for o, v in opts.items():
        lg.check(lg.gemm_set_option(o, v))
    try:
        fn()
    finally:
        for o, v in old.items():
            lg.gemm_set_option(o, v)


TMA_SHAPES = [(4, 4, 1), (128, 128, 16), (130, 257, 7), (261, 132, 95), (516, 389, 333),
              (1000, 1003, 1100)]


@pytest.mark.parametrize("shape", TMA_SHAPES)
@pytest.mark.parametrize("cm", (0, 1))
def test_sgemm_tma_fed(shape, cm):
    M, N, K = shape

    def body():
        run_and_check(M, N, K, lg.GEMM_F32, 1, 1, cm, dist="pm1", seed=M + K,
                      lda_pad=pad4(M), ldb_pad=pad4(N) + 4)
        run_and_check(M, N, K, lg.GEMM_F32, 1, 1, cm, dist="int", seed=M + N,
                      lda_pad=pad4(M) + 8, ldb_pad=pad4(N), ldc_pad=1)
    with_options({lg.GEMM_OPT_SIMT_CONFIG: 9}, body)


@pytest.mark.parametrize("am,bm,cm", [(0, 0, 1), (0, 1, 0), (1, 0, 1), (0, 0, 0)])
def test_sgemm_tma_fed_after_transpose(am, bm, cm):
    # K-major operands reach the TMA path through the transpose pre-pass
    # (MN-major copies with pitches rounded up to 4 elements)
    def body():
        run_and_check(301, 163, 97, lg.GEMM_F32, am, bm, cm, dist="pm1", seed=51,
                      lda_pad=3, ldb_pad=1, ldc_pad=2)
        run_and_check(64, 96, 33, lg.GEMM_F32, am, bm, cm, dist="int", seed=52)
    with_options({lg.GEMM_OPT_SIMT_CONFIG: 9, lg.GEMM_OPT_SIMT_TRANSPOSE: 2}, body)


@pytest.mark.parametrize("cm", (0, 1))
def test_sgemm_tma_fed_split_tail_forced(cm):
    # every last-wave tile cut into K-slices: slices of one k-tile, and empty
    # slices (no copies, no waits) on the shortest K
    def body():
        for i, (M, N, K) in enumerate([(4, 4, 1), (16, 20, 7), (132, 260, 300),
                                       (260, 132, 33)]):
            run_and_check(M, N, K, lg.GEMM_F32, 1, 1, cm, dist="int", seed=60 + i,
                          lda_pad=pad4(M), ldb_pad=pad4(N), ldc_pad=i % 3)
        run_and_check(300, 520, 200, lg.GEMM_F32, 1, 1, cm, dist="pm1", seed=65)
    with_options({lg.GEMM_OPT_SIMT_CONFIG: 9, lg.GEMM_OPT_SIMT_SPLIT_TAIL: 2}, body)


@pytest.mark.parametrize("M,N,K", [(2557, 2043, 1100), (1000, 1001, 1100)])
@pytest.mark.parametrize("am,bm", [(0, 0), (1, 1)])
def test_sgemm_split_tail_automatic(am, bm, M, N, K):
    # 2557 x 2043: 320 tiles on 152 SMs, two full rounds and 16 tail tiles;
    # 1000 x 1001: 64 tiles, no full round. With 69 k-tiles the automatic
    # rule cuts the tail into 2 slices in both.
    assert lg.gemm_get_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL) == 0
    run_and_check(M, N, K, lg.GEMM_F32, am, bm, 1, dist="int", seed=46)
