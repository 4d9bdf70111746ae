"""The phase-trace build of the tensor-core kernel (libgemm_trace.so, compiled
with LIBGEMM_TC_TRACE): a registered device buffer receives %globaltimer
stamps at fixed points of every role, 64 per CTA. One traced call must stamp
every CTA in order (entry <= set-up done <= exit, the first unit's MMAs
start before they end, the epilogue ends before the CTA exits) and still
match the oracle. Built here once, loaded in a child process."""

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

CHILD = textwrap.dedent("""
    import ctypes, sys
    sys.path.insert(0, {tests!r}); sys.path.insert(0, {root!r})
    import numpy as np, torch
    import dense_gemm_06_gb300 as lg
    from dense_gemm_06_gb300 import _build
    lib = lg.load(_build.LIB_TRACE)
    raw = ctypes.CDLL(_build.LIB_TRACE)
    raw.libgemm_tc_trace_buffer.argtypes = [ctypes.c_void_p]
    from test_parity_1_small import run_and_check
    buf = torch.zeros(1024 * 64, dtype=torch.int64, device="cuda")
    raw.libgemm_tc_trace_buffer(buf.data_ptr())
    try:
        # 2048 x 2048 x 1024 fp16 -> fp32: 64 pair tiles, one unit per pair
        run_and_check(2048, 2048, 1024, lg.GEMM_F16_F32, 0, 0, 1, "int", 3, cta_group=2)
    finally:
        raw.libgemm_tc_trace_buffer(None)
    t = buf.cpu().numpy().reshape(1024, 64)
    ctas = np.nonzero(t[:, 0])[0]
    assert len(ctas) >= 64, len(ctas)
    t = t[ctas]
    assert np.all(t[:, 1] >= t[:, 0]) and np.all(t[:, 63] >= t[:, 1]), "set-up / exit order"
    lead = t[(t[:, 4] > 0)]
    assert len(lead) >= 32, len(lead)
    assert np.all(lead[:, 5] >= lead[:, 4]), "MMA end before its start"
    epi = t[(t[:, 62] > 0)]
    assert len(epi) >= 64 and np.all(epi[:, 63] >= epi[:, 62]), "epilogue after exit"
    print("ctas", len(ctas), "kernel us", round(float(t[:, 63].max() - t[:, 0].min()) / 1000, 1))
""")


def test_trace_build_stamps_every_phase_in_order():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dense_gemm_06_gb300 import _build
    _build.build(trace=True)
    r = subprocess.run([sys.executable, "-c", CHILD.format(tests=TESTS, root=ROOT)], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "ctas" in r.stdout
