"""Host-side logic of bench.py on the CPU: the throughput arithmetic, the
single-GPU argument rule, the clock-record summary, the peaks and the
source-keyed traffic record."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_throughput():
    f = 5 * 2.0 * 8192 ** 3
    one = bench.throughput_tflops(f, 10, 680.0)
    assert one == pytest.approx(f * 10 / 0.68 / 1e12)
    assert bench.throughput_tflops(f, 20, 680.0) == pytest.approx(2 * one)


@pytest.mark.parametrize("impl", ["native", "reference"])
def test_only_one_gpu_is_accepted(impl):
    # the library is single-GPU: any other --gpus is refused before anything runs
    for n in (0, 2, 8):
        with pytest.raises(SystemExit) as e:
            bench.main(["--impl", impl, "--gpus", str(n), "--steps", "1", "--warmup", "0"])
        assert e.value.code == 2


def test_no_process_group_code_left():
    # no torch.distributed / NCCL path remains in the benchmark
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert "torch.distributed" not in src and "init_process_group" not in src


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

