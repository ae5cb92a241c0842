"""The tensor-core path's cluster split-K mode.  Where the tiles are too few
to fill the SMs, each tile runs on one thread-block cluster of S CTAs, each
taking an equal part of the tile's k-steps; the CTAs add up their partial
sums through distributed shared memory, in rank order, and store.  Parity
against the oracle over cluster sizes, ragged shapes, every format, both
weight layouts and the fused epilogues.  The plan is read back from the
library's debug line, so a silent fallback to another mode fails the test."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import assert_parity, check_full, check_sampled, oracle_ref, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture
def csk(monkeypatch, capfd):
    """Sets the cluster split-K policy; returns a reader of the last plan."""
    monkeypatch.setenv("WQ_DEBUG", "1")

    def use(setting):
        monkeypatch.setenv("WQ_TC_CSK", str(setting))
        capfd.readouterr()

    def plan():
        err = capfd.readouterr().err
        lines = [ln for ln in err.splitlines() if ln.startswith("wq: tcgen05")]
        assert lines, err[-400:]
        return lines[-1]

    use.plan = plan
    return use


def grid_of(line):
    return int(line.rsplit("grid=", 1)[1])


@pytest.mark.parametrize("fmt", ["int4", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K", [(128, 1024, 3072), (100, 3072, 3072), (17, 384, 4096), (256, 1000, 1024),
                                   (64, 200, 640), (160, 1152, 2048)])
def test_auto(fmt, M, N, K, csk):
    csk(1)
    group = 64 if (fmt == "int4" and K % 128) else None
    p = synth.make_problem(fmt, M, N, K, group=group, seed=M + N + K)
    check_full(p, "fp32", path="tc", what=f"{fmt} {M}x{N}x{K} cluster split-K")
    line = csk.plan()
    assert "cluster split-K" in line, line


@pytest.mark.parametrize("S", [2, 3, 4, 5, 6, 7, 8])
def test_each_cluster_size(S, csk):
    """Forced S: the k-steps split S ways (K = 3072: 48 k-steps, uneven for
    S = 5 and 7), and each CTA reduces an uneven share of the column groups."""
    csk(S)
    p = synth.make_problem("int4", 96, 640, 3072, seed=S)
    check_full(p, "fp32", path="tc", what=f"S={S}")
    line = csk.plan()
    assert "cluster split-K" in line and grid_of(line) == 5 * S, line


def test_more_ctas_than_k_steps(csk):
    """K = 128: two k-steps, so at most two CTAs per tile."""
    csk(8)
    p = synth.make_problem("nvfp4", 40, 256, 128, seed=3)
    check_full(p, "fp32", path="tc", what="K=128")
    line = csk.plan()
    assert "cluster split-K" in line and grid_of(line) == 2 * 2, line


@pytest.mark.parametrize("layer", ["q", "kv", "gate_up", "down"])
def test_decoder_layers_m128(layer, csk):
    csk(1)
    p = synth.layer_problem(layer, 128)
    check_sampled(p, "bf16", k=16, path="tc", what=f"{layer} M=128 cluster split-K")
    assert "cluster split-K" in csk.plan()


def test_prepacked(csk):
    csk(1)
    p = synth.make_problem("int4", 128, 3072, 3072, seed=9)
    A, packed, scales, zeros = to_dev(p)
    pre = wq.prepack(packed, scales, zeros, "int4")
    C = wq.gemm_prepacked(A, pre, out_dtype="fp32", path="tc")
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    assert "cluster split-K" in csk.plan()
    Ce, S = oracle_ref(p)
    assert_parity(C.cpu().numpy().astype(np.float64), Ce, S, "fp32", "prepacked cluster split-K")


@pytest.mark.parametrize("gated", [False, True])
def test_epilogues(gated, csk):
    csk(1)
    p = synth.make_problem("int4", 72, 768, 2048, seed=31)
    rng = np.random.default_rng(31)
    N = p["N"]
    bias = synth.bf16_bits((rng.normal(size=N) * 0.5).astype(np.float32))
    res = synth.bf16_bits(rng.normal(size=(p["M"], N // 2 if gated else N)).astype(np.float32))
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    A, packed, scales, zeros = to_dev(p)
    Y = wq.gemm(A, packed, scales, zeros, "int4", out_dtype="fp32", path="tc", bias=dev(bias), residual=dev(res),
                gated=gated)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    assert "cluster split-K" in csk.plan()
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], "int4", 128)
    Ye, T = oracle.epilogue(C, S, bias, res, gated, "fp32")
    err = np.abs(Y.cpu().numpy().astype(np.float64) - Ye)
    assert (err <= T).all(), float(np.max(err - T))


def test_repeated_calls_bit_identical(csk):
    """The sums run in a fixed order: the same call gives the same bits."""
    csk(1)
    p = synth.make_problem("int4", 128, 1024, 3072, seed=12)
    A, packed, scales, zeros = to_dev(p)
    first = wq.gemm(A, packed, scales, zeros, "int4", out_dtype="fp32", path="tc")
    for _ in range(50):
        again = wq.gemm(A, packed, scales, zeros, "int4", out_dtype="fp32", path="tc")
        assert torch.equal(first, again)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK


def test_off_keeps_the_other_plans(csk):
    """With the mode off, the same shape runs whole tiles (no workspace)."""
    csk(0)
    p = synth.make_problem("int4", 128, 1024, 3072, seed=13)
    check_full(p, "fp32", path="tc", what="cluster split-K off")
    assert "data-parallel" in csk.plan()
