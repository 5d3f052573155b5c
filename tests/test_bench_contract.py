"""bench.py's reference arm (the oracle on the host cores) prints one JSON line with the
keys the benchmark contract asks for. Runs on CPU with the 256 x 256 toy workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "toy_256", "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    r = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert k in r, k
    assert r["impl"] == "reference" and r["steps"] == 2 and r["warmup"] == 1 and r["n_gpus"] == 1
    assert r["value"] > 0 and r["unit"] == "Mweights/s" and r["higher_is_better"] is True
    assert r["config"]["workload"] == "toy_256" and (r["config"]["m"], r["config"]["d"]) == (256, 256)
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == r["value"]
    e2e = r["e2e"]
    assert e2e["value"] == r["value"] and e2e["unit"] == r["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
