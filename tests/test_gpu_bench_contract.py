"""bench.py on the GPU: one short run of the default line, checked against the
line's contract (every key, its type and the relations between them)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_default_line_keeps_the_contract():
    d = _run("--steps", "200", "--warmup", "3", "--cpu-seconds", "1")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 200 and d["warmup"] >= 3
    assert d["higher_is_better"] is False and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1e3 - d["value"]) < 1e-2
    assert "workload" in d["config"] and "l2" in d["config"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert r["traffic"] is None or r["traffic"] > 0.9 * r["algorithmic_bytes"]
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    e = d["e2e"]
    # the copies overlap the neighbouring steps' kernels: e2e is at least about the kernels' time
    assert e["value"] >= 0.97 * d["value"] and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["serial_value"] >= 0.97 * e["value"]
    assert d["gpu_launches"] >= d["steps"]
    assert d["clocks"]["sm_mhz"] > 0 and isinstance(d["clocks"]["reasons"], list)


@pytest.mark.parametrize("args", [("--op", "prepare"), ("--workload", "4", "--part", "a", "--dcp-ranks", "2"),
                                  ("--query-tokens", "2"), ("--kv", "fp8")])
def test_other_lines_run(args):
    d = _run(*args, "--steps", "100", "--warmup", "3", "--no-cpu-baseline", "--no-e2e")
    assert d["value"] > 0 and d["roofline"]["achieved"] > 0
