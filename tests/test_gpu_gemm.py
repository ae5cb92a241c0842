"""GEMM parity on the GPU: wq_gemm / wq_gemm_ex against the oracle.

Every output element is checked against the oracle's exact fp64 result with
the method's gate.  The workloads are the seeded synthetic inputs of
weight_only_bit_w4a16_gb300.synth at their full sizes (sampled rows and
columns where the oracle would take too long for every element), ragged
shapes around every tile edge, exact invariants (one-hot activations, sign
flip, power-of-two scale, zero weights) and determinism.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import (assert_parity, check_full, check_sampled, gpu_gemm, oracle_ref, to_dev)

pytestmark = pytest.mark.gpu


# -- the workloads at full size ------------------------------------------------
def test_tiny_nvfp4_fp32_out():
    p = synth.workload_problem("tiny_nvfp4")
    check_full(p, "fp32", what="tiny_nvfp4")
    check_full(p, "fp32", path="gemv", what="tiny_nvfp4 gemv")


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("seed", [0, 1])
def test_decode_int4(M, seed):
    p = synth.workload_problem("decode_int4", M=M, seed=seed)
    check_full(p, "bf16", what=f"decode_int4 M={M}")


def test_prefill_mxfp4():
    p = synth.workload_problem("prefill_mxfp4")
    check_sampled(p, "bf16", what="prefill_mxfp4")


def test_large_nvfp4():
    """8192^3 NVFP4: 64 random rows (all 8192 columns) and 64 random columns
    (all 8192 rows), plus the first and last of each, against the oracle."""
    p = synth.workload_problem("large_nvfp4")
    check_sampled(p, "bf16", k=64, what="large_nvfp4")


@pytest.mark.parametrize("layer", list(synth.LAYER_SHAPES))
@pytest.mark.parametrize("M", [1, 16, 128, 2048])
def test_layer_sweep(layer, M):
    """Every decoder projection at every M, the LM head at M = 2048 (a 0.5 GB
    output, checked on the sampled rows and columns copied from the device)
    included."""
    p = synth.layer_problem(layer, M)
    check_sampled(p, "bf16", k=8, what=f"{layer} M={M}")


# -- both kernels on the same shapes ------------------------------------------
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
@pytest.mark.parametrize("path", ["gemv", "auto"])
@pytest.mark.parametrize("M", [1, 5, 8, 9, 16, 17, 40, 128, 300])
def test_paths_agree_with_oracle(fmt, path, M):
    p = synth.make_problem(fmt, M, 384, 1024, seed=M)
    out = "fp32" if M % 2 else "bf16"
    check_full(p, out, path=path, what=f"{fmt} M={M} {path}")


# -- ragged shapes ---------------------------------------------------------------
@pytest.mark.parametrize("M", list(range(1, 18)) + [127, 129])
def test_ragged_M(M):
    p = synth.make_problem("int4", M, 200, 640, seed=100 + M)
    check_full(p, "fp32", what=f"ragged M={M}")


@pytest.mark.parametrize("N", [1, 7, 15, 16, 17, 100, 257, 1000])
@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
def test_ragged_N(N, fmt):
    for M in (3, 16, 200):
        p = synth.make_problem(fmt, M, N, 512, seed=N + M)
        check_full(p, "bf16", what=f"{fmt} N={N} M={M}")


@pytest.mark.parametrize("K", [32, 64, 96, 160, 1056, 4160])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_ragged_K(K, fmt):
    for M in (2, 130):
        p = synth.make_problem(fmt, M, 96, K, seed=K + M)
        check_full(p, "fp32", what=f"{fmt} K={K} M={M}")


@pytest.mark.parametrize("group", [32, 64, 96, 128, 256])
def test_int4_group_sizes(group):
    K = 768
    for M in (4, 64):
        p = synth.make_problem("int4", M, 160, K, group=group, seed=group)
        check_full(p, "fp32", what=f"int4 g{group} M={M}")


def test_zero_K_gives_zeros():
    dev = torch.device("cuda:0")
    A = torch.zeros((4, 0), dtype=torch.bfloat16, device=dev)
    packed = torch.zeros((8, 0), dtype=torch.uint8, device=dev)
    scales = torch.zeros((8, 0), dtype=torch.uint8, device=dev)
    C = torch.full((4, 8), 5.0, device=dev)
    st = wq.wq_gemm_ex(A.data_ptr() or 0x10000, packed.data_ptr() or 0x10000, scales.data_ptr() or 0x10000,
                       None, C.data_ptr(), 4, 8, 0, wq.WQ_NVFP4 | wq.WQ_OUT_F32, 16,
                       torch.cuda.current_stream().cuda_stream, wq.WQ_PATH_AUTO)
    torch.cuda.synchronize()
    assert st == wq.WQ_OK
    assert torch.all(C == 0)


# -- exact invariants (fp32 output) ---------------------------------------------
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
@pytest.mark.parametrize("path", ["gemv", "auto"])
def test_one_hot_activation_selects_weight(fmt, path):
    K = 512
    p = synth.make_problem(fmt, 1, 64, K, seed=3)
    ks = np.array([0, 1, 2, 31, 32, 127, 128, 300, 511] + list(range(40, 80)))
    A = np.zeros((len(ks), K), dtype=np.uint16)
    A[np.arange(len(ks)), ks] = 0x3F80
    p["A"], p["M"] = A, len(ks)
    C = gpu_gemm(p, "fp32", path)
    W64, Wb = oracle.dequant(p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    w64 = W64[:, ks].T
    wbf = np.asarray(
        torch.from_numpy(Wb[:, ks].T.astype(np.int16).copy()).view(torch.bfloat16).float().numpy(),
        dtype=np.float64)
    # fp4 weights are exact in bf16; int4 weights are either exact (scale
    # applied in fp32 after the MMA) or their bf16 image
    assert np.all((C == w64) | (C == wbf))
    if fmt != "int4":
        assert np.array_equal(C, w64)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("M", [3, 200])
def test_sign_flip_negates_exactly(fmt, M):
    p = synth.make_problem(fmt, M, 128, 512, seed=7)
    C = gpu_gemm(p, "fp32")
    q = dict(p, packed=p["packed"] ^ 0x88)
    C2 = gpu_gemm(q, "fp32")
    assert np.array_equal(C2, -C)


@pytest.mark.parametrize("M", [3, 200])
def test_mxfp4_exponent_plus_one_doubles_exactly(M):
    p = synth.make_problem("mxfp4", M, 128, 512, seed=8)
    C = gpu_gemm(p, "fp32")
    C2 = gpu_gemm(dict(p, scales=p["scales"] + 1), "fp32")
    assert np.array_equal(C2, 2 * C)


@pytest.mark.parametrize("M", [4, 64])
def test_int4_codes_equal_zero_give_zero(M):
    N, K, g = 96, 512, 128
    rng = np.random.default_rng(5)
    z = rng.integers(0, 16, size=(N, K // g), dtype=np.uint8)
    codes = np.repeat(z, g, axis=1)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    p = synth.make_problem("int4", M, N, K, seed=5)
    p.update(packed=packed, zeros=z)
    assert np.all(gpu_gemm(p, "fp32") == 0)


def test_nvfp4_zero_scale_gives_zero():
    p = synth.make_problem("nvfp4", 40, 64, 256, seed=6)
    p["scales"] = np.zeros_like(p["scales"])
    assert np.all(gpu_gemm(p, "fp32") == 0)


# -- determinism, streams, output bounds ---------------------------------------
@pytest.mark.parametrize("M", [16, 256])
def test_deterministic(M):
    p = synth.make_problem("int4", M, 1024, 3072, seed=9)
    C1 = gpu_gemm(p, "fp32")
    C2 = gpu_gemm(p, "fp32")
    assert np.array_equal(C1, C2)


def test_side_stream_and_guard_region():
    p = synth.make_problem("nvfp4", 12, 72, 256, seed=10)
    A, packed, scales, zeros = to_dev(p)
    buf = torch.full((12 * 72 + 256,), 3.0, device="cuda")
    C = buf[: 12 * 72].view(12, 72)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        wq.gemm(A, packed, scales, zeros, "nvfp4", out_dtype="fp32", out=C)
    s.synchronize()
    assert torch.all(buf[12 * 72:] == 3.0)
    Ce, S = oracle_ref(p)
    assert_parity(C.cpu().numpy().astype(np.float64), Ce, S, "fp32", "side stream")


# -- launch options -------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["int4", "nvfp4"])
def test_inputs_ready_chain(fmt):
    """WQ_LAUNCH_INPUTS_READY on the input layout: calls whose activations were
    written before the chain read them at once and wait for their
    predecessor only before storing; a dependent call and a plain stream
    consumer afterwards see every output complete and oracle-green."""
    N, K = 1024, 3072
    dev = torch.device("cuda:0")
    ps = [synth.make_problem(fmt, M, N, K, seed=60 + i) for i, M in enumerate((1, 4, 16, 2))]
    ins = [to_dev(p) for p in ps]
    torch.cuda.synchronize()
    outs = [wq.gemm(A, pk, sc, zr, fmt, inputs_ready=True) for A, pk, sc, zr in ins]
    q = synth.make_problem(fmt, 2, N, N, seed=69)
    _, pk2, sc2, zr2 = to_dev(q)
    torch.cuda.synchronize()
    outs = [wq.gemm(A, pk, sc, zr, fmt, inputs_ready=True) for A, pk, sc, zr in ins]
    y = wq.gemm(outs[-1], pk2, sc2, zr2, fmt, overlap=True)   # reads the last ready call's output
    total = sum(o.float().sum() for o in outs)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    for p, o in zip(ps, outs):
        Ce, S = oracle_ref(p)
        assert_parity(o.float().cpu().numpy().astype(np.float64), Ce, S, "bf16", f"{fmt} ready chain")
    Ce, S = oracle_ref(dict(q, A=outs[-1].view(torch.int16).cpu().numpy().view(np.uint16)))
    assert_parity(y.float().cpu().numpy().astype(np.float64), Ce, S, "bf16", f"{fmt} dependent after ready")
    assert float(total) == float(sum(o.float().sum() for o in outs))


def test_overlapped_launches_chain_correctly():
    """WQ_LAUNCH_OVERLAP: calls on one stream, each reading the previous
    call's output as its activations, must still see that output complete."""
    K = N = 1024
    ps = [synth.make_problem("int4", 4, N, K, seed=40 + i) for i in range(3)]
    dev = torch.device("cuda:0")
    x = torch.from_numpy(ps[0]["A"].view(np.int16)).view(torch.bfloat16).to(dev)
    outs = []
    for p in ps:
        _, packed, scales, zeros = to_dev(p)
        x = wq.gemm(x, packed, scales, zeros, "int4", overlap=True)
        outs.append(x)
    torch.cuda.synchronize()
    # replay on the host, step by step, through the oracle
    a_bits = ps[0]["A"]
    for p, o in zip(ps, outs):
        q = dict(p, A=a_bits)
        Ce, S = oracle_ref(q)
        got = o.float().cpu().numpy().astype(np.float64)
        assert_parity(got, Ce, S, "bf16", "overlap chain")
        a_bits = o.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_cluster_kernel_variant(M, monkeypatch):
    """The cluster-split GEMV (used for large M x K) on the decode shape."""
    monkeypatch.setenv("WQ_GEMV_FORCE_CLUSTER", "1")
    p = synth.workload_problem("decode_int4", M=M, seed=3)
    check_full(p, "bf16", path="gemv", what=f"cluster M={M}")
    q = synth.make_problem("nvfp4", M, 512, 1024, seed=M)
    check_full(q, "fp32", path="gemv", what=f"cluster nvfp4 M={M}")


@pytest.mark.parametrize("wk", ["0", "1", "2", "3", "4"])
def test_split_kernel_warp_splits(wk, monkeypatch):
    """Every K split of the register-streaming split kernel gives the same parity."""
    monkeypatch.setenv("WQ_GEMV_KERNEL", "split")
    monkeypatch.setenv("WQ_GEMV_WK_LOG2", wk)
    for fmt, M in (("int4", 1), ("int4", 12), ("mxfp4", 3)):
        p = synth.make_problem(fmt, M, 300, 3072, seed=int(wk) + M)
        check_full(p, "fp32", path="gemv", what=f"{fmt} wk={wk} M={M}")


@pytest.mark.parametrize("rb,wk", [("1", "0"), ("1", "2"), ("1", "3"), ("2", "1"), ("2", "3"), ("4", "0"),
                                   ("4", "2"), ("8", "1")])
def test_streaming_kernel_cta_shapes(rb, wk, monkeypatch):
    """Every CTA shape of the TMA-streaming GEMV (16-row blocks per CTA x warps
    splitting K) gives the same parity, on ragged N and K and on every mode."""
    monkeypatch.setenv("WQ_GEMV_RB", rb)
    monkeypatch.setenv("WQ_GEMV_TMA_WK", wk)
    cases = (("int4", 1, 300, 3072, 128), ("int4", 12, 200, 1024, 128), ("int4", 5, 70, 640, 64),
             ("nvfp4", 3, 130, 544, 16), ("mxfp4", 16, 100, 2080, 32))
    for fmt, M, N, K, g in cases:
        p = synth.make_problem(fmt, M, N, K, group=g, seed=int(rb) * 10 + int(wk) + M)
        check_full(p, "fp32", path="gemv", what=f"{fmt} rb={rb} wk={wk} M={M} N={N} K={K}")


# -- the second exact decode step: int4 zero points above 128, MXFP4 E > 142 --
@pytest.mark.parametrize("path", ["gemv", "auto"])
@pytest.mark.parametrize("M", [3, 16, 96])
@pytest.mark.parametrize("group", [128, 64])
def test_int4_zero_points_above_128(path, M, group):
    p = synth.make_problem("int4", M, 144, 1024, group=group, seed=M + group)
    rng = np.random.default_rng(M)
    z = p["zeros"].copy()
    big = rng.random(z.shape) < 0.3
    z[big] = rng.integers(129, 256, size=int(big.sum()), dtype=np.uint8)
    p["zeros"] = z
    check_full(p, "fp32", path=path, what=f"int4 big zeros g{group} M={M} {path}")


@pytest.mark.parametrize("path", ["gemv", "auto"])
@pytest.mark.parametrize("M", [3, 16, 96])
def test_mxfp4_scales_above_2_pow_15(path, M):
    p = synth.make_problem("mxfp4", M, 144, 1024, seed=M)
    rng = np.random.default_rng(M)
    E = p["scales"].copy()
    big = rng.random(E.shape) < 0.3
    E[big] = rng.integers(143, 161, size=int(big.sum()), dtype=np.uint8)
    p["scales"] = E
    check_full(p, "fp32", path=path, what=f"mxfp4 E>142 M={M} {path}")
