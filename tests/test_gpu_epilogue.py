"""Fused epilogues on the GPU (wq_gemm_fused): bias per weight row, the
SiLU-gated product of an interleaved gate/up pair, bf16 residual -- on the
small-M kernels and the tensor-core kernel (whole tiles and stream-K split
tiles), against the oracle's fp64 epilogue and its tolerance."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import to_dev

pytestmark = pytest.mark.gpu


def bits_to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run(p, bias, res, gated, out, path="auto", workspace=None):
    A, packed, scales, zeros = to_dev(p)
    C = wq.gemm(A, packed, scales, zeros, p["fmt"], p["group"], out_dtype=out, path=path, workspace=workspace,
                bias=None if bias is None else bits_to_dev(bias),
                residual=None if res is None else bits_to_dev(res), gated=gated)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    return C.float().cpu().numpy().astype(np.float64)


def check(p, bias, res, gated, out, path="auto", workspace=None, what=""):
    Y = run(p, bias, res, gated, out, path, workspace)
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], p["fmt"], p["group"])
    Ye, T = oracle.epilogue(C, S, bias, res, gated, out)
    err = np.abs(Y - Ye)
    bad = ~(err <= T)
    assert not bad.any(), f"{what}: {int(bad.sum())}/{Y.size} outside; worst {np.max(err - T):.3e}"


def inputs(p, gated, seed):
    rng = np.random.default_rng(seed)
    N = p["N"]
    bias = synth.bf16_bits((rng.normal(size=N) * 0.5).astype(np.float32))
    res = synth.bf16_bits(rng.normal(size=(p["M"], N // 2 if gated else N)).astype(np.float32))
    return bias, res


@pytest.mark.parametrize("fmt", ["int4", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M", [1, 4, 16, 40, 200])
def test_gated_with_bias_and_residual(fmt, M):
    p = synth.make_problem(fmt, M, 256, 1024, seed=M)
    bias, res = inputs(p, True, M)
    out = "fp32" if M % 2 else "bf16"
    check(p, bias, res, True, out, what=f"{fmt} M={M} gated+bias+res")


@pytest.mark.parametrize("M", [1, 16, 130])
@pytest.mark.parametrize("parts", ["bias", "res", "gated"])
def test_each_part_alone(M, parts):
    p = synth.make_problem("int4", M, 160, 768, seed=M + 3)
    bias, res = inputs(p, parts == "gated", M)
    check(p, bias if parts == "bias" else None, res if parts == "res" else None, parts == "gated", "fp32",
          what=f"M={M} {parts}")


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("kernel", ["split", "cluster"])
def test_register_streaming_kernels(M, kernel, monkeypatch):
    monkeypatch.setenv("WQ_GEMV_KERNEL", kernel)
    p = synth.make_problem("int4", M, 128, 1024, seed=M + 11)
    bias, res = inputs(p, True, M)
    check(p, bias, res, True, "fp32", path="gemv", what=f"{kernel} M={M}")


def test_gate_up_decode_shape():
    """The decoder's fused gate/up projection at batch 1: 2 x 8192 weight rows,
    K = 3072, output 8192."""
    p = synth.make_problem("int4", 1, 16384, 3072, seed=21)
    bias, res = inputs(p, True, 21)
    check(p, None, None, True, "bf16", what="gate_up M=1")
    check(p, bias, res, True, "bf16", what="gate_up M=1 bias+res")


@pytest.mark.parametrize("M", [128, 300])
def test_stream_k_owner_applies_the_epilogue(M, monkeypatch):
    monkeypatch.setenv("WQ_TC_CSK", "0")   # stream-K, not the cluster split of these few tiles
    p = synth.make_problem("int4", M, 512, 4096, seed=M + 5)
    ws = wq.workspace(M, 512, 4096, "int4")
    assert ws is not None
    bias, res = inputs(p, True, M)
    check(p, bias, res, True, "fp32", path="tc", workspace=ws, what=f"stream-K M={M}")
