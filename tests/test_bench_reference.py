"""bench.py's reference arm (the CPU oracle timed on this host) keeps the JSON
contract: one line with the arm's metric, unit, value, the oracle as
`cpu_baseline`, an `e2e` object with zero copied bytes; under torchrun only
rank 0 runs and prints.  CPU only, a bounded sample (about ten seconds)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    return p.stdout


def test_reference_arm_json_line():
    out = run(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    lines = [l for l in out.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"].startswith("fused Q4_K SwiGLU-MLP") and d["unit"] == "tok/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["warmup"] >= 3
    assert d["config"]["name"] == "prefill_T2048" and d["config"]["T"] == 2048
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    out = run(["--impl", "reference", "--steps", "1", "--warmup", "0"],
              {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.strip() == ""
