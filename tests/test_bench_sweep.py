"""Host logic of the bench's decoder-layer sweep (CPU only): the calls of a
step cover every projection of the 3B decoder and the tied LM head at every
M, and a call's roofline bound is the larger of its two closed forms."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0}


def test_sweep_calls_cover_the_decoder():
    w = bench.BENCH_WORKLOADS["layer_sweep"]
    shapes = bench.sweep_shapes(w)
    assert shapes == {"q": (3072, 3072), "k": (1024, 3072), "v": (1024, 3072), "o": (3072, 3072),
                      "gate": (8192, 3072), "up": (8192, 3072), "down": (3072, 8192), "lm_head": (128256, 3072)}
    assert tuple(w["Ms"]) == (1, 16, 128, 2048)
    assert w["fmt"] == "int4" and w["group"] == 128 and w["out"] == "bf16"


def test_roofline_time_decode_is_bytes():
    # M = 1 on the gate shape: A 6144 B + codes 12582912 + bf16 scales and
    # zeros 3 B per 128-group (589824) + C 16384 B, at 8 TB/s
    t, bound = bench.roofline_time(1, 8192, 3072, PEAKS)
    assert bound == "hbm"
    assert abs(t - (6144 + 12582912 + 589824 + 16384) / 8e12) < 1e-15


def test_roofline_time_prefill_is_flops():
    # M = 2048 on the LM head: 2 M N K flops at 2 PFLOP/s
    t, bound = bench.roofline_time(2048, 128256, 3072, PEAKS)
    assert bound == "tensor"
    assert abs(t - 2 * 2048 * 128256 * 3072 / 2e15) < 1e-12


def test_roofline_time_takes_the_larger_bound():
    # M = 128 on q: 2 * 128 * 3072^2 = 2.42 GFLOP (1.21 us at 2 PF) against
    # 0.79 + 4.94 + 0.79 MB of A, weights and C (0.82 us at 8 TB/s)
    t, bound = bench.roofline_time(128, 3072, 3072, PEAKS)
    assert bound == "tensor" and abs(t - 2 * 128 * 3072 * 3072 / 2e15) < 1e-15


def test_both_arms_describe_the_same_workload():
    """The config of a line names the workload only, so our arm and the
    reference arm build the same dict (how our arm launches and lays out its
    weights goes under "setup")."""
    import inspect
    for name in bench.BENCH_WORKLOADS:
        cfg = bench.bench_config(name, 1)
        assert cfg["workload"] == name and cfg["parallelism"] == "replicas x1"
        assert {"format", "group", "M", "out", "calls_per_step"} <= set(cfg)
    src_ours, src_ref = inspect.getsource(bench.run_ours), inspect.getsource(bench.run_reference)
    assert '"config": bench_config(args.workload, ws)' in src_ours
    assert '"config": bench_config(args.workload, ws)' in src_ref
    assert bench.bench_config("decode_int4", 1) == {
        "workload": "decode_int4", "format": "int4", "group": 128, "M": [1, 4, 16], "out": "bf16",
        "N": 8192, "K": 3072, "calls_per_step": 3, "parallelism": "replicas x1"}
