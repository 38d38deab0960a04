"""The benchmark's JSON line, checked on the CPU through its reference arm
(the float64 oracle on host cores, a small sample): every key of the line
exists with the right type, and ranks other than 0 print nothing."""
import json
import os
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent


def run_bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], cwd=ROOT, env=e, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    return out.stdout


def test_reference_arm_line_has_every_key():
    lines = [l for l in run_bench("--impl", "reference", "--steps", "2", "--warmup", "1",
                                  "--ref-budget", "3").splitlines() if l.strip()]
    d = json.loads(lines[-1])
    assert d["impl"] == "reference"
    for key, typ in [("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)]:
        assert isinstance(d[key], typ), key
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["vs_baseline"] is None
    assert "workload" in d["config"] and "sample" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    out = run_bench("--impl", "reference", "--steps", "1", "--warmup", "1", "--ref-budget", "1",
                    env={"RANK": "1", "WORLD_SIZE": "2"})
    assert out.strip() == ""


def test_bench_reads_nothing_from_outside_the_repository():
    """bench.py names no absolute path: every file it reads is found relative
    to the repository (the measured peaks, the profiles, the oracle)."""
    import re
    text = (ROOT / "bench.py").read_text()
    assert not re.findall(r"""["']/[A-Za-z]""", text)
