"""bench.py asked for more than one GPU: the path is built for one GPU, so rank 0 prints
one line that says the run is unavailable and every rank exits 0 before touching CUDA;
the reference arm does its work on rank 0 only. Runs on the CPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=120, cwd=ROOT, env=env)


def test_two_gpus_asked_prints_unavailable_line():
    out = _run(["--gpus", "2", "--steps", "1", "--warmup", "3"], {})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    r = json.loads(lines[0])
    assert r["n_gpus"] == 2 and "single-GPU" in r["unavailable"]
    assert "value" not in r


def test_torchrun_ranks_other_than_zero_print_nothing():
    out = _run(["--gpus", "2"], {"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""
    out0 = _run(["--gpus", "2"], {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert out0.returncode == 0 and "unavailable" in json.loads(out0.stdout.strip())


def test_rate_counts_every_step():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rate_mweights(4, 1000, 2.0) == 4 * 1000 / 2.0 / 1e6


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(bench.argparse.Namespace(workload="llama_4096_g128", layer=0, steps=1, warmup=1, gpus=2,
                                                 threads=None, tokens=None))
    assert capsys.readouterr().out == ""
