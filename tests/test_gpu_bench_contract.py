"""bench.py's output line, as its readers expect it.

Runs the benchmark as a user would (a child process, small step counts) and
checks the one JSON line it prints: the keys and their types, a positive
throughput, the roofline and CPU-baseline objects, the end-to-end object
with its copied bytes, the count of the library's launches and the clock
record; and the reference arm's line on the same workload."""
import json
import os
import subprocess
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_our_line_has_every_key():
    d = run_bench("--workload", "tiny", "--steps", "5", "--warmup", "3", "--clock-preroll", "0.2")
    for key, typ in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("roofline", dict), ("e2e", dict),
                     ("gpu_launches", int), ("clocks", dict)):
        assert isinstance(d.get(key), typ), (key, d.get(key))
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["n_gpus"] == 1
    assert d["steps"] == 5 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert "workload" in d["config"] and d["config"]["shard_params"] == 1_836_288
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) <= 1e-9 * r["frac"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] >= 2 * d["config"]["shard_params"]
    assert e["d2h_bytes_per_step"] >= 2 * d["config"]["shard_params"]
    # the library's kernels in the timed region: two a step on a flat shard
    assert d["gpu_launches"] == 2 * d["steps"]
    c = d["clocks"]
    assert c["sm_mhz"] > 0 and c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)


def test_reference_arm_line():
    """The reference arm times the oracle on the same workload: its config
    names the same workload and shard as ours."""
    import bench
    d = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3")
    assert d["impl"] == "reference"
    assert d["config"]["workload"] == bench.TITLES["tiny"] and d["config"]["shard_params"] == 1_836_288
    assert d["value"] > 0 and d["unit"] == "params/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
