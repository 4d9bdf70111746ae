"""The dispatch log (GEMM_LOG=1): one stderr line per decision a call takes,
silent when the variable is unset. The library reads the variable once, so
each case runs in a child process."""

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import torch
    import dense_gemm_06_gb300 as lg
    lg.load()
    M, N, K = 512, 384, 256
    a = torch.zeros(M * K, dtype=torch.int16, device="cuda")
    b = torch.zeros(N * K, dtype=torch.int16, device="cuda")
    c = torch.zeros(M * N, dtype=torch.float32, device="cuda")
    lg.check(lg.gemm(M, N, K, a, K, 0, b, K, 0, c, N, 1, lg.GEMM_F16_F32))
    x = torch.zeros(256 * 256, dtype=torch.float32, device="cuda")
    y = torch.zeros_like(x)
    lg.check(lg.gemm(256, 256, 256, x, 256, 1, x, 256, 1, y, 256, 1, lg.GEMM_F32))
    torch.cuda.synchronize()
""")


def _run(env_value):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    env = dict(os.environ)
    env.pop("GEMM_LOG", None)
    if env_value is not None:
        env["GEMM_LOG"] = env_value
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stderr.splitlines() if ln.startswith("libgemm: ")]


def test_log_names_each_kernel_and_its_plan():
    lines = _run("1")
    tc = [ln for ln in lines if "tcgen05 512x384x256" in ln]
    ffma = [ln for ln in lines if ln.startswith("libgemm: FFMA SGEMM") and "256x256x256" in ln]
    assert len(tc) == 1 and "tiles" in tc[0] and "units" in tc[0], lines
    assert len(ffma) == 1 and "tiles of 128 x 128" in ffma[0], lines


@pytest.mark.parametrize("value", [None, "0", ""])
def test_log_off_by_default(value):
    assert _run(value) == []
