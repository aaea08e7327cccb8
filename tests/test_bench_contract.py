"""The benchmark's reference arm (the FP64 oracle on the host cores, the only other
implementation of this path) runs on CPU: launched as the driver launches it, it prints one
JSON line with the keys the benchmark contract names, and its own cpu_baseline and e2e."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert "workload" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_decode_traffic_figure_matches_the_kernel_sources():
    """bench.py's roofline.traffic for decode B=256 is one ncu capture of the decode kernel; it
    stands only for the sources it was taken on. When they change, take the capture again (ncu
    dram__bytes_read.sum and dram__bytes_write.sum of one B=256 decode launch) and record the
    new bytes and the new source hash in bench.py."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.decode_sources_sha256() == bench.DEC_TRAFFIC_SRC_SHA256, (
        "the decode kernel's sources changed since its DRAM traffic was captured")
