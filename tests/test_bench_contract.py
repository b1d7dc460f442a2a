"""The benchmark's reference arm (the fp64 oracle on the host cores) runs without a GPU
and prints the one JSON line the benchmark contract asks for."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--ref-budget", "0.2", "--workload", "prefill_1k"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3
    assert d["config"]["workload"] == "prefill_1k"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "2"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_stored_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    """roofline.traffic comes from one ncu capture: bench.py reports it only while the kernel's
    source hashes to the value stored with it, and null for any other source."""
    sys.path.insert(0, ROOT)
    import bench
    nbytes, sha = bench.DOMINANT_TRAFFIC["prefill_4k"]
    assert nbytes > 0 and len(sha) == 16
    src = tmp_path / "kernel.cu"
    src.write_bytes(open(bench.DOMINANT_SRC, "rb").read())
    monkeypatch.setattr(bench, "DOMINANT_SRC", str(src))
    expect = nbytes if bench.source_sha16(str(src)) == sha else None
    assert bench.dominant_traffic("prefill_4k") == expect
    src.write_bytes(open(bench.DOMINANT_SRC, "rb").read() + b"\n// changed\n")
    assert bench.dominant_traffic("prefill_4k") is None
    assert bench.dominant_traffic("varlen_64") is None
