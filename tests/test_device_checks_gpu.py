"""The debug build with device-side checks (libgemm_checks.so, compiled with
LIBGEMM_DEVICE_CHECKS): every kernel path runs parity cases against the
oracle through it, and no device-side check may fail (tensor-core work units
inside the tile grid, 16-byte aligned TMA coordinates, every epilogue store
inside C, FFMA tiles and K-slices inside the problem, every FFMA store inside
C). The build is made here, once, and loaded in a child process."""

import os
import subprocess
import sys
import textwrap

import pytest

import dense_gemm_06_gb300 as lg

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

CHILD = textwrap.dedent("""
    import itertools, sys
    sys.path.insert(0, {tests!r}); sys.path.insert(0, {root!r})
    import dense_gemm_06_gb300 as lg
    from dense_gemm_06_gb300 import _build
    lg.load(_build.LIB_CHECKS)
    from test_parity_1_small import TC_MODES, run_and_check
    n = 0
    # tensor cores: every CTA mode and scheduler, every operand major, ragged
    # tails in M, N and K; misaligned pitches (repack, scalar C stores)
    for mode, (cg, mc, sch) in sorted(TC_MODES.items()):
        for am, bm in itertools.product((0, 1), (0, 1)):
            run_and_check(257, 513, 1037, lg.GEMM_F16_F32, am, bm, 1, "int", 1037,
                          cta_group=cg, multicast=mc, scheduler=sch); n += 1
        run_and_check(333, 277, 131, lg.GEMM_F16_F32, 0, 1, 1, "int", 6, lda_pad=1,
                      ldb_pad=3, ldc_pad=1, cta_group=cg, multicast=mc, scheduler=sch); n += 1
        run_and_check(333, 277, 131, lg.GEMM_BF16_BF16, 1, 0, 0, "normal", 7, lda_pad=5,
                      ldb_pad=1, ldc_pad=3, cta_group=cg, multicast=mc, scheduler=sch); n += 1
        run_and_check(384, 520, 640, lg.GEMM_F16_F16, 0, 1, 1, "int", 5, cta_group=cg,
                      tc_store=1, multicast=mc, scheduler=sch); n += 1
    # unit widths and the last round's half-width units
    for cg, tile_n in ((1, 64), (1, 128), (2, 128), (2, 256)):
        run_and_check(4736, 2304, 192, lg.GEMM_F16_F32, 0, 1, 1, "int", 13, cta_group=cg,
                      tile_n=tile_n, split=2); n += 1
    # FFMA: every tile configuration, ragged shapes, padded pitches
    for cfg in range(1, 10):
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, cfg))
        for am, bm in itertools.product((0, 1), (0, 1)):
            run_and_check(257, 131, 33, lg.GEMM_F32, am, bm, 1, "pm1", 11); n += 1
        run_and_check(200, 150, 90, lg.GEMM_F32, 1, 1, 0, "int", 3, lda_pad=3, ldb_pad=5,
                      ldc_pad=1); n += 1
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_CONFIG, 0))
    # FFMA K-slices and stream-K, forced
    for split, shape in ((2, (300, 520, 2000)), (3, (1000, 1001, 333)), (3, (2048, 2048, 256))):
        lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, split))
        run_and_check(*shape, lg.GEMM_F32, 1, 1, 1, "int", shape[2]); n += 1
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_SIMT_SPLIT_TAIL, 0))
    rc, first = lg.gemm_device_checks()
    assert rc == lg.GEMM_OK, rc
    assert first == 0, f"device-side check failed: code {{first >> 56}}, detail {{first & ((1 << 56) - 1):#x}}"
    print("cases", n)
""")


def test_checks_build_passes_every_path():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dense_gemm_06_gb300 import _build
    _build.build(checks=True)
    r = subprocess.run([sys.executable, "-c", CHILD.format(tests=TESTS, root=ROOT)], cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "cases" in r.stdout
