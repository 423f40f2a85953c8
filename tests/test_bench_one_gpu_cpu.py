"""bench.py drives one GPU: asked for more (--gpus N, or several torchrun
ranks), rank 0 prints one `unavailable` line and every rank exits 0 without
touching a GPU (the prefill kernels multicast K/V gathers inside clusters,
which the library does for one GPU's own memory only)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(args, env_extra):
    env = dict(os.environ, **env_extra)
    env["CUDA_VISIBLE_DEVICES"] = ""  # a run that reached for a GPU would fail
    res = subprocess.run([sys.executable, "bench.py"] + args, cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    return [ln for ln in res.stdout.splitlines() if ln.strip()]


def test_two_gpus_are_refused_on_rank_zero():
    lines = run(["--gpus", "2"], {"RANK": "0"})
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2 and "one GPU" in rec["unavailable"]
    assert "value" not in rec


def test_torchrun_ranks_are_refused_and_silent_off_rank_zero():
    lines = run(["--gpus", "2"], {"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"})
    assert len(lines) == 1 and "unavailable" in json.loads(lines[0])
    assert run(["--gpus", "2"], {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
