"""bench.py's reference arm on the host (no GPU): one JSON line with the keys
the benchmark contract names, the oracle timed on the tiny workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert cb["host"]["logical_cpus"] >= 1
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_dominant_kernel_traffic_record_matches_its_sources():
    """The DRAM traffic bench.py reports for the prefill step's dominant kernel
    was captured on the sources as they are now (a change to them without a
    new capture turns the record off, and this test red)."""
    sys.path.insert(0, ROOT)
    import bench
    rec = bench.DOMINANT_TRAFFIC[("k_pack_permute", "prefill")]
    assert bench.dominant_traffic("k_pack_permute", "prefill") == rec["bytes"]
    # the capture sits a little below the kernel's HBM bytes (x partly in L2)
    assert 0.95 * 479.4e6 < rec["bytes"] <= 479.4e6
