"""bench.py's reference arm (the fp64 oracle on the host cores) runs without a
GPU: its JSON line carries the keys and units the benchmark contract fixes,
with the step's own metric, and an end-to-end entry that moves no bytes."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    import bench

    d = _run("--impl", "reference", "--config", "tiny_causal", "--steps", "2", "--warmup", "1")
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny_causal"
    assert "leading 256 x 256 block" in d["config"]["sample"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert set(cb) == {"kind", "cores", "sample", "value", "unit"}
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_document_sample():
    d = _run("--impl", "reference", "--config", "doc_packing", "--steps", "1", "--warmup", "0")
    assert d["config"]["sample"] == "the first document of head 0 per step"
    assert "the first document of head 0" in d["cpu_baseline"]["sample"]
