"""bench.py on the GPU, end to end, on the small workload: one JSON line with
the contract's keys, a roofline object, clocks, the pipelined e2e figure
whose delivered results match the same step run alone, and the oracle
baseline beside it."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

pytestmark = pytest.mark.gpu


def run(argv):
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(argv)
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1, buf.getvalue()
    return json.loads(lines[0])


@pytest.mark.parametrize("layout", ["prepacked", "plain"])
def test_bench_line_tiny(layout):
    d = run(["--workload", "tiny_nvfp4", "--steps", "64", "--warmup", "3", "--cpu-budget", "0.05",
             "--layout", layout])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "gpu_launches", "e2e",
                "cpu_baseline"):
        assert key in d, key
    assert d["steps"] == 64 and d["warmup"] == 3 and d["value"] > 0 and d["gpu_launches"] == 64
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["achieved"] > 0 and r["peak"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["results_checked"] is True
    assert e["h2d_bytes_per_step"] == 16 * 512 * 2 and e["d2h_bytes_per_step"] == 16 * 256 * 4
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
