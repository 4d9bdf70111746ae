"""Builds libgemm.so from csrc/ with nvcc for sm_103a only (no cmake).

Each translation unit compiles in parallel into _build/, with the ptxas
resource report (registers, spills, shared memory) kept beside each object;
the objects link into dense_gemm_06_gb300/libgemm.so against the shared CUDA
runtime (so the library shares the runtime PyTorch already loaded).

build(checks=True) compiles the debug build with device-side checks
(-DLIBGEMM_DEVICE_CHECKS: tile coordinates, TMA coordinates and store
addresses checked in the kernels, see gemm_device_checks in gemm.h) into
_build_checks/ and libgemm_checks.so; build(trace=True) the phase-trace
build of the tensor-core kernel (-DLIBGEMM_TC_TRACE: %globaltimer stamps at
fixed points of every role, 64 per CTA, into a device buffer registered with
the extra export libgemm_tc_trace_buffer(void*)) into _build_trace/ and
libgemm_trace.so. The default build has neither.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgemm.so")
BUILD_CHECKS = os.path.join(HERE, "_build_checks")
LIB_CHECKS = os.path.join(HERE, "libgemm_checks.so")
CHECKS_FLAGS = ["-DLIBGEMM_DEVICE_CHECKS"]
BUILD_TRACE = os.path.join(HERE, "_build_trace")
LIB_TRACE = os.path.join(HERE, "libgemm_trace.so")
TRACE_FLAGS = ["-DLIBGEMM_TC_TRACE"]
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", INCLUDE]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else (shutil.which("nvcc") or "nvcc")


def _cuda_lib_dir() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return os.path.join(cuda, "lib64")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, force: bool, out_dir: str = BUILD, extra=()) -> str:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    log = obj[:-2] + ".ptxas.txt"
    if not force and os.path.exists(obj) and \
            os.path.getmtime(obj) >= max(os.path.getmtime(src), _deps_mtime()):
        return obj
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj + ".tmp"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stderr[-6000:]}")
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, jobs: int | None = None, checks: bool = False,
          trace: bool = False) -> str:
    """Compile every csrc/*.cu for sm_103a and link libgemm.so (checks: the
    debug build with device-side checks, libgemm_checks.so; trace: the
    phase-trace build, libgemm_trace.so); returns its path."""
    if checks and trace:
        raise ValueError("one debug variant at a time")
    out_dir, lib, extra = BUILD, LIB, []
    if checks:
        out_dir, lib, extra = BUILD_CHECKS, LIB_CHECKS, CHECKS_FLAGS
    elif trace:
        out_dir, lib, extra = BUILD_TRACE, LIB_TRACE, TRACE_FLAGS
    os.makedirs(out_dir, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, force, out_dir, extra), srcs))
    newest = max(os.path.getmtime(o) for o in objs)
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < newest:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath," + _cuda_lib_dir()]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr[-6000:]}")
        os.replace(tmp, lib)
    return lib


def ptxas_report() -> str:
    """The ptxas resource lines of the last build (registers, spills, smem)."""
    out = []
    for f in sorted(glob.glob(os.path.join(BUILD, "*.ptxas.txt"))):
        with open(f) as fh:
            out.append(fh.read())
    return "\n".join(out)


if __name__ == "__main__":
    print(build(force=True))
