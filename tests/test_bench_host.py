"""bench.py's host-side logic on CPU: the DRAM-traffic figure is taken from the
committed ncu summary only while the GEMM kernel sources match the digest it
was measured on, and the reference arm's JSON line keeps the contract's keys."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    digest = bench.kernel_source_digest()
    assert len(digest) == 64
    summary = tmp_path / "traffic.md"
    summary.write_text("sources_sha256: %s\nbytes_per_launch: 123456\n" % digest)
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(summary))
    assert bench.measured_traffic() == 123456
    summary.write_text("sources_sha256: %s\nbytes_per_launch: 123456\n" % ("0" * 64))
    assert bench.measured_traffic() is None  # another build: no figure
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(tmp_path / "missing.md"))
    assert bench.measured_traffic() is None


def test_committed_traffic_summary_matches_these_sources():
    # the committed summaries were captured on the kernel sources in this tree
    assert bench.measured_traffic() is not None
    assert bench.measured_traffic("mx") is not None
    assert bench.measured_traffic("tensor") is not None


def test_each_recipe_digest_covers_its_own_kernel():
    assert bench.kernel_source_digest("mx") != bench.kernel_source_digest("tensor")
    assert "gemm_mx.cu" in bench.RECIPE_SOURCES["mx"] and "gemm_tensor.cu" in bench.RECIPE_SOURCES["tensor"]
    assert "gemm_kernel.cuh" in bench.RECIPE_SOURCES["mx"]  # the shared epilogues


def test_reference_arm_line(tmp_path):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_bias_gradient_modes(monkeypatch):
    # the step's default takes db in dZ's transposed cast; every mode is accepted
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    assert bench.parse_args().bias_grad == "cast"
    for mode in ("cast", "dgrad", "operand"):
        monkeypatch.setattr(sys, "argv", ["bench.py", "--bias-grad", mode])
        assert bench.parse_args().bias_grad == mode
    from fp8_linear_layer_gb300.linear import LinearTrainStep, MxLinearTrainStep
    import inspect
    assert inspect.signature(LinearTrainStep.__init__).parameters["bias_grad"].default == "cast"
    assert inspect.signature(MxLinearTrainStep.__init__).parameters["bias_grad"].default == "cast"
