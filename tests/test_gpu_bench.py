"""bench.py's JSON line on a short run with the smaller workloads: every key
of the contract is there and consistent (the rates follow from the times
and the counted work, the rooflines from their peaks, one step is one direct
launch, the binning launches and one brick launch), in the default mode and
with the map shared as z-slabs."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def _bench(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
           "--direct-workload", "direct_3d", "--cutoff-workload", "cutoff_uniform", "--cpu-seconds", "0.4",
           "--no-msm", "--no-secondary", *extra]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("mode", [(), ("--shard-map",)])
def test_bench_line_contract(mode):
    d = _bench(*mode)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["dtype"] == "f32"
    assert d["scaling"] == ("strong" if mode else "weak")
    assert "128x128x64" in d["config"]["workload"] and "capacity 0" in d["config"]["workload"]
    # value = pairs of the step / mean direct time
    assert d["value"] == pytest.approx(d["config"]["direct"]["pairs"] / (d["direct"]["ms"] * 1e-3), rel=1e-9)
    r = d["roofline"]
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9) and 0.2 < r["frac"] < 1.2
    c = d["cutoff"]
    assert c["pairs_per_step"]["useful"] <= c["pairs_per_step"]["evaluated"] <= c["pairs_per_step"]["examined"]
    assert c["ms"] == pytest.approx(c["ms_binning"] + c["ms_map"], rel=1e-9)
    assert 0.0 < c["roofline_map"]["frac"] < 1.2 and 0.0 < c["roofline_binning"]["frac"] < 1.0
    # 3 timed steps, each one direct launch, the binning launches and one brick launch
    assert d["gpu_launches"] % 3 == 0 and 7 <= d["gpu_launches"] // 3 <= 8
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
