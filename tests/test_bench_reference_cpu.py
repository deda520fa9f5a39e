"""The bench's reference arm (the float64 oracle on host cores) prints the
contract's JSON line on rank 0 and nothing on the other ranks; it needs no
GPU, so it runs here."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"}


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
           "--warmup", "3", "--ref-seqs", "4"]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("tiny")


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_all_cores_oracle_pass_uses_every_core_and_cleans_up():
    # The bench's second CPU figure: the oracle over the same sample on a
    # spawn pool with one single-threaded process per host core.
    import glob
    import tempfile
    sys.path.insert(0, ROOT)
    import bench
    before = set(glob.glob(os.path.join(tempfile.gettempdir(), "pk_oracle_pool_*")))
    r = bench.run_cpu_oracle_pool("tiny", 0, 4, 0.3)
    assert r["cores"] == len(os.sched_getaffinity(0))
    assert r["seqs"] == 4 and r["bytes"] > 0 and len(r["times"]) >= 1 and min(r["times"]) > 0
    assert set(glob.glob(os.path.join(tempfile.gettempdir(), "pk_oracle_pool_*"))) == before
