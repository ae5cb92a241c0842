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


def test_bench_default_decode_line():
    """The default workload as the driver runs it (--steps 20 --warmup 5):
    the headline with the calls' inputs declared ready, the other launch
    modes and the per-M times beside it, and the tensor-core block (prefill,
    8192^3 and one decoder-layer sweep step) with its own clocks."""
    d = run(["--steps", "20", "--warmup", "5", "--cpu-budget", "0.05"])
    assert d["config"]["workload"] == "decode_int4" and d["config"]["M"] == [1, 4, 16]
    assert d["steps"] == 20 and d["gpu_launches"] == 60 and d["value"] > 0
    assert "INPUTS_READY" in d["setup"]["launch"]
    assert set(d["other_launch_modes"]) == {"overlap", "plain"}
    for M in ("1", "4", "16"):
        pm = d["per_m"][M]
        assert pm["us_per_call"] > 0 and pm["overlap"]["us_per_call"] > 0
    tc = d["tensor_core"]
    for name in ("prefill_mxfp4", "large_nvfp4"):
        r = tc[name]["roofline"]
        assert r["bound"] == "tensor" and 0 < r["frac"] < 1.5 and tc[name]["clocks"] is not None
    assert tc["large_nvfp4"]["M"] == tc["large_nvfp4"]["N"] == tc["large_nvfp4"]["K"] == 8192
    assert tc["layer_sweep_step"]["calls"] == 32 and tc["layer_sweep_step"]["pct_of_roofline"] > 0
