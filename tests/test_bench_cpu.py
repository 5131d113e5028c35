"""The benchmark's reference arm (the oracle on a bounded sample) runs on the
CPU and prints the one JSON line of the contract."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--cpu-budget", "1"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "dtype",
                "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["M"] == 4096 and d["config"]["N"] == 14336 and d["config"]["K"] == 4096


def test_profile_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """bench.py reports a profile's dram traffic only while the hash of the
    kernel's sources recorded with it matches the sources (else null)."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "fp8_scaled_quantization_quantize_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("// kernel v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = hashlib.sha256(b"// kernel v1\n").hexdigest()
    (prof / "p.json").write_text(json.dumps({"traffic_bytes_per_launch": 12345, "sources_sha256": digest}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.sources_sha256(("k.cu",)) == digest
    assert bench.measured_traffic("p.json", ("k.cu",)) == 12345.0
    (src / "k.cu").write_text("// kernel v2\n")
    assert bench.measured_traffic("p.json", ("k.cu",)) is None
    assert bench.measured_traffic("missing.json", ("k.cu",)) is None

