"""Host-side logic of bench.py on the CPU: the replica path's barrier and
max-over-ranks timing on a world-size-2 gloo group, the whole-job
throughput, the reference arm's rank handling and the clock-record summary."""

import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slow = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
        bench.barrier(world)
        q.put((rank, slow))
    finally:
        dist.destroy_process_group()


def test_two_rank_barrier_and_max_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]   # every rank sees the slowest rank's time


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    bench.barrier(1)


def test_throughput_is_weak_scaling_over_replicas():
    f = 5 * 2.0 * 8192 ** 3
    one = bench.throughput_tflops(f, 10, 1, 680.0)
    two = bench.throughput_tflops(f, 10, 2, 680.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(f * 10 / 0.68 / 1e12)


def test_reference_arm_rank_nonzero_exits_quietly(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert buf.getvalue() == ""


def test_clock_summary():
    lines = ["2070, 2070, 900.1, Not Active, Not Active, Not Active, Not Active\n",
             "1950, 2070, 1399.0, Not Active, Not Active, Not Active, Active\n",
             "2010, 2070, 1300.0, Not Active, Not Active, Not Active, Not Active\n",
             "garbage line\n"]
    c = bench.summarize_clocks(lines)
    assert c["sm_mhz"] == 2010 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert bench.summarize_clocks([]) is None


def test_peaks_file_or_fallback():
    peaks, src = bench.load_peaks()
    assert src in ("measured", "fallback")
    assert peaks["bf16_tflops"] > 1000 and peaks["hbm_gbs"] > 1000
    assert bench.FFMA_PEAK_TFLOPS == pytest.approx(152 * 128 * 2 * 2.07 / 1e3)
    tf, how = bench.ffma_peak(152, 2070.0)
    assert tf == pytest.approx(80.55, abs=0.01) and "queried" in how
    tf, how = bench.ffma_peak(None, None)  # nothing queried: GB300's figures
    assert tf == pytest.approx(bench.FFMA_PEAK_TFLOPS) and "assumed" in how
    assert bench.ffma_peak(148, 1965.0)[0] == pytest.approx(148 * 128 * 2 * 1.965 / 1e3)


def test_traffic_entry_needs_matching_source(tmp_path, monkeypatch):
    # the per-launch DRAM bytes of a kernel are only reported while the
    # kernel's source is the one the ncu counters were taken on
    import hashlib
    src_dir = tmp_path / "dense_gemm_06_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (src_dir / "k.cu").write_text("// kernel v1\n")
    digest = hashlib.sha256(b"// kernel v1\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    entry = {"bytes_per_launch": 123, "source": "k.cu", "source_sha256_16": digest}
    (prof / "traffic.json").write_text(json.dumps({"k": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k") == 123
    (src_dir / "k.cu").write_text("// kernel v2\n")
    assert bench.profiled_traffic("k") is None
    assert bench.profiled_traffic("missing") is None


def test_traffic_entry_over_several_sources(tmp_path, monkeypatch):
    # a kernel spread over several files is keyed on all of them, in order
    import hashlib
    src_dir = tmp_path / "dense_gemm_06_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (src_dir / "k.cuh").write_text("// kernel\n")
    (src_dir / "helpers.cuh").write_text("// helpers v1\n")
    digest = hashlib.sha256(b"// kernel\n// helpers v1\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    entry = {"bytes_per_launch": 456, "source": ["k.cuh", "helpers.cuh"],
             "source_sha256_16": digest}
    (prof / "traffic.json").write_text(json.dumps({"k": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k") == 456
    (src_dir / "helpers.cuh").write_text("// helpers v2\n")  # either file changing
    assert bench.profiled_traffic("k") is None
    (src_dir / "helpers.cuh").write_text("// helpers v1\n")
    (src_dir / "k.cuh").unlink()                              # or going missing
    assert bench.profiled_traffic("k") is None

