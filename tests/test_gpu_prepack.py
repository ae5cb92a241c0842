"""The prepacked weight path on the GPU: wq_prepack writes the same bytes as
the oracle's layout writer, and wq_gemm_prepacked computes C = A . deq(B)^T
within the method's gate against the oracle on the ORIGINAL (unpacked)
weight -- every format, ragged N / K / M, the rare second decode steps,
fused epilogues, chained launches and the decode configuration's full size."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import prepack as opk
import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import assert_parity, host_rows_cols, oracle_ref, sample, to_dev

pytestmark = pytest.mark.gpu


def prepack_dev(p):
    _, packed, scales, zeros = to_dev(p)
    pre = wq.prepack(packed, scales, zeros, p["fmt"], p["group"])
    torch.cuda.synchronize()
    return pre


def run_pre(p, out="fp32", overlap=False, pre=None, ready=False, **epi):
    A, _, _, _ = to_dev(p)
    pre = pre or prepack_dev(p)
    C = wq.gemm_prepacked(A, pre, out_dtype=out, overlap=overlap, inputs_ready=ready, **epi)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    return C.float().cpu().numpy().astype(np.float64)


def check_pre(p, out="fp32", overlap=False, what="", ready=False):
    C = run_pre(p, out, overlap, ready=ready)
    Ce, S = oracle_ref(p)
    assert_parity(C, Ce, S, out, what)
    return C


# -- the repack itself -----------------------------------------------------------
@pytest.mark.parametrize("fmt,N,K", [
    ("int4", 20, 256), ("int4", 37, 384), ("int4", 300, 3072),
    ("nvfp4", 20, 256), ("nvfp4", 33, 160), ("nvfp4", 130, 544),
    ("mxfp4", 20, 256), ("mxfp4", 5, 96), ("mxfp4", 100, 2080),
])
def test_prepack_bytes_equal_oracle(fmt, N, K):
    p = synth.make_problem(fmt, 1, N, K, seed=N + K)
    if fmt == "int4":   # full uint8 zero points, the second subtrahend included
        rng = np.random.default_rng(K)
        p["zeros"] = rng.integers(0, 256, p["zeros"].shape, dtype=np.uint8)
    pre = prepack_dev(p)
    want = opk.prepack(p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    got = pre.buf.cpu().numpy()
    assert got.size == want.size
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


# -- the GEMM on prepacked weights ------------------------------------------------
# Two small-M kernels read the layout: the ring kernel (calls that declare
# their inputs ready) and the staged kernel (dependent and plain calls).
# WQ_GEMV_PRE_KERNEL forces one; the ring runs here with its inputs declared
# ready, as it is launched in use.
@pytest.fixture(params=["staged", "ring"])
def kernel(request, monkeypatch):
    monkeypatch.setenv("WQ_GEMV_PRE_KERNEL", request.param)
    return request.param


def ready_for(kernel):
    return kernel == "ring"


@pytest.mark.parametrize("fmt", ["int4", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 17, 40])
def test_parity_against_oracle(fmt, M, kernel):
    p = synth.make_problem(fmt, M, 256, 1024, seed=M)
    check_pre(p, "fp32" if M % 2 else "bf16", what=f"{kernel} {fmt} M={M}", ready=ready_for(kernel))


@pytest.mark.parametrize("fmt,N,K", [("int4", 200, 384), ("int4", 8, 128), ("nvfp4", 130, 544),
                                     ("nvfp4", 33, 160), ("mxfp4", 100, 2080), ("mxfp4", 5, 96)])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_ragged_shapes(fmt, N, K, M, kernel):
    """N not a multiple of 16; fp4 K not a multiple of 128 (a partial last
    block whose activation tail the kernel zeroes)."""
    p = synth.make_problem(fmt, M, N, K, seed=N + M)
    check_pre(p, "fp32", what=f"{kernel} {fmt} N={N} K={K} M={M}", ready=ready_for(kernel))


@pytest.mark.parametrize("rb,wk", [("1", "0"), ("1", "3"), ("2", "1"), ("4", "2"), ("8", "1")])
def test_staged_cta_shapes(rb, wk, monkeypatch):
    monkeypatch.setenv("WQ_GEMV_PRE_KERNEL", "staged")
    monkeypatch.setenv("WQ_GEMV_RB", rb)
    monkeypatch.setenv("WQ_GEMV_TMA_WK", wk)
    for fmt, M, N, K in (("int4", 1, 300, 3072), ("int4", 12, 200, 1024), ("nvfp4", 3, 130, 544),
                         ("mxfp4", 16, 100, 2080)):
        p = synth.make_problem(fmt, M, N, K, seed=int(rb) * 10 + int(wk) + M)
        # a forced shape that cannot hold its slice is refused: at most 16
        # blocks of 128 k per warp, at most 227 KB of shared memory
        nk = -(-K // 128)
        ipw = -(-nk // (1 << int(wk)))
        warps = int(rb) << int(wk)
        rec = 96 if fmt == "int4" else 512   # int4 reserves 96 B per block (48 used)
        # activation rows per CTA: 16 when they fit, else 8, 4, 2, 1
        fits = [256 + warps * ipw * (1024 + rec) + min(M, mr) * (nk * 256 + 64) + 128 <= 227 * 1024
                for mr in (16, 8, 4, 2, 1)]
        if ipw > 16 or not any(fits):
            with pytest.raises(wq.WQError) as e:
                run_pre(p, "fp32")
            assert e.value.status == wq.WQ_ERR_UNSUPPORTED
            continue
        check_pre(p, "fp32", what=f"{fmt} rb={rb} wk={wk} M={M}")


def _ring_smem(fmt, M, K, RB, Wk, P):
    """Shared memory of a forced CTA shape of the ring kernel: the layout its
    source documents (barriers, a ring of P slots per warp of RB code blocks
    + the activation rows, the records, and the partial sums that alias
    them)."""
    r128 = lambda x: (x + 127) // 128 * 128  # noqa: E731
    nk = -(-K // 128)
    ipw = -(-nk // Wk)
    P = min(P, ipw)
    mrows = 16 if M > 8 else 8
    Mc, MP = min(M, mrows), (16 if M > 8 else 8)
    ring_off = r128(8 * Wk * P)
    slot = r128(1024 * RB + 256 * Mc)
    end = ring_off + Wk * P * slot + Wk * RB * ipw * (96 if fmt == "int4" else 512)   # int4: 96 reserved
    red = ring_off + Wk * MP * (RB * 16 + 4) * 4
    return max(end, red) + 128


@pytest.mark.parametrize("rb,wk,ring", [("1", "0", "3"), ("1", "3", "2"), ("2", "1", "3"), ("4", "2", "4"),
                                        ("4", "0", "1"), ("2", "3", "5")])
def test_ring_cta_shapes(rb, wk, ring, monkeypatch):
    """Every forced shape of the ring kernel (row blocks per CTA, warps, ring
    slots) computes the product; a shape above 227 KB of shared memory is
    refused."""
    monkeypatch.setenv("WQ_RING_RB", rb)
    monkeypatch.setenv("WQ_RING_WK", wk)
    monkeypatch.setenv("WQ_RING_P", ring)
    for fmt, M, N, K in (("int4", 1, 300, 3072), ("int4", 12, 200, 1024), ("nvfp4", 3, 130, 544),
                         ("mxfp4", 16, 100, 2080), ("nvfp4", 2, 40, 16384)):
        p = synth.make_problem(fmt, M, N, K, seed=int(rb) * 10 + int(wk) + M)
        if _ring_smem(fmt, M, K, int(rb), 1 << int(wk), int(ring)) > 227 * 1024:
            with pytest.raises(wq.WQError) as e:
                run_pre(p, "fp32", ready=True)
            assert e.value.status == wq.WQ_ERR_UNSUPPORTED
            continue
        check_pre(p, "fp32", what=f"{fmt} rb={rb} wk={wk} ring={ring} M={M}", ready=True)


def test_ring_shape_refusal_is_reachable():
    """The shape table above really contains a refused case (fp4 records of
    16384 k in one warp of 4 row blocks)."""
    assert _ring_smem("nvfp4", 2, 16384, 4, 1, 1) > 227 * 1024
    assert _ring_smem("int4", 1, 3072, 2, 2, 3) < 64 * 1024


@pytest.mark.parametrize("M", [3, 16])
def test_int4_zero_points_above_128(M, kernel):
    p = synth.make_problem("int4", M, 144, 1024, seed=M + 7)
    rng = np.random.default_rng(M)
    z = p["zeros"].copy()
    big = rng.random(z.shape) < 0.3
    z[big] = rng.integers(129, 256, size=int(big.sum()), dtype=np.uint8)
    p["zeros"] = z
    check_pre(p, "fp32", what=f"{kernel} int4 big zeros M={M}", ready=ready_for(kernel))


@pytest.mark.parametrize("M", [3, 16])
def test_int4_zero_points_up_to_128(M, kernel):
    """Zero points 0, 1, 127 and 128 only: the prepacked flag stays 0 and every
    subtrahend is the one-step 128 + z (z = 128 carries into the exponent)."""
    p = synth.make_problem("int4", M, 144, 1024, seed=M + 11)
    rng = np.random.default_rng(M + 1)
    p["zeros"] = rng.choice(np.array([0, 1, 127, 128], np.uint8), size=p["zeros"].shape)
    pre = prepack_dev(p)
    assert int(pre.buf[-16].item()) == 0
    check_pre(p, "fp32", what=f"{kernel} int4 zeros <= 128 M={M}", ready=ready_for(kernel))
    if M == 16:
        C = run_tc(p)
        Ce, S = oracle_ref(p)
        assert_parity(C, Ce, S, "fp32", "tc int4 zeros <= 128")


@pytest.mark.parametrize("M", [3, 16])
def test_mxfp4_scales_above_2_pow_15(M, kernel):
    p = synth.make_problem("mxfp4", M, 144, 1024, seed=M + 9)
    rng = np.random.default_rng(M)
    E = p["scales"].copy()
    big = rng.random(E.shape) < 0.3
    E[big] = rng.integers(143, 161, size=int(big.sum()), dtype=np.uint8)
    p["scales"] = E
    check_pre(p, "fp32", what=f"{kernel} mxfp4 E>142 M={M}", ready=ready_for(kernel))


@pytest.mark.parametrize("M", [4, 16])
def test_int4_codes_equal_zero_give_zero(M, kernel):
    N, K, g = 96, 512, 128
    rng = np.random.default_rng(5)
    z = rng.integers(0, 16, size=(N, K // g), dtype=np.uint8)
    codes = np.repeat(z, g, axis=1)
    p = synth.make_problem("int4", M, N, K, seed=5)
    p.update(packed=(codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), zeros=z)
    assert np.all(run_pre(p, "fp32", ready=ready_for(kernel)) == 0)


@pytest.mark.parametrize("fmt", ["int4", "nvfp4"])
def test_one_hot_activation_selects_weight(fmt, kernel):
    """a[m, k] = 1 at one k per row: C[m, n] = w[n, k] exactly (fp32 out)."""
    N, K = 64, 512
    p = synth.make_problem(fmt, 16, N, K, seed=11)
    ks = np.array([0, 1, 7, 8, 31, 64, 127, 128, 129, 200, 255, 300, 383, 384, 500, 511])
    A = np.zeros((16, K), np.float32)
    A[np.arange(16), ks] = 1.0
    p["A"] = synth.bf16_bits(A)
    W64, _ = oracle.dequant(p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    C = run_pre(p, "fp32", ready=ready_for(kernel))
    assert np.array_equal(C, W64[:, ks].T)


def test_deterministic_and_overlap_equal():
    p = synth.make_problem("int4", 16, 1024, 3072, seed=9)
    pre = prepack_dev(p)
    C1 = run_pre(p, "fp32", pre=pre)
    C2 = run_pre(p, "fp32", pre=pre)
    C3 = run_pre(p, "fp32", overlap=True, pre=pre)
    assert np.array_equal(C1, C2) and np.array_equal(C1, C3)


def test_ring_deterministic_across_launch_flags(monkeypatch):
    """The ring kernel with a forced shape gives the same bits whether it is
    launched plain, overlapped or with its inputs declared ready."""
    monkeypatch.setenv("WQ_GEMV_PRE_KERNEL", "ring")
    monkeypatch.setenv("WQ_RING_RB", "2")
    monkeypatch.setenv("WQ_RING_WK", "1")
    p = synth.make_problem("int4", 16, 1024, 3072, seed=9)
    pre = prepack_dev(p)
    C1 = run_pre(p, "fp32", pre=pre)
    C2 = run_pre(p, "fp32", pre=pre, ready=True)
    C3 = run_pre(p, "fp32", pre=pre, overlap=True)
    C4 = run_pre(p, "fp32", pre=pre, ready=True)
    assert np.array_equal(C1, C2) and np.array_equal(C1, C3) and np.array_equal(C2, C4)


def test_inputs_ready_chain():
    """A chain of calls with WQ_LAUNCH_INPUTS_READY (activations written
    before the chain, distinct weights, M = 1, 4, 16 in turn, then dependent
    calls and a plain torch consumer): each call completes in stream order,
    so every output read after the chain is complete and oracle-green."""
    N, K = 1024, 3072
    ps = [synth.make_problem("int4", M, N, K, seed=70 + i) for i, M in enumerate((1, 4, 16, 1, 4, 16))]
    pres = [prepack_dev(p) for p in ps]
    As = [to_dev(p)[0] for p in ps]
    torch.cuda.synchronize()
    outs = []
    for A, pre in zip(As, pres):
        outs.append(wq.gemm_prepacked(A, pre, inputs_ready=True))
    # a dependent call that reads the last ready call's output as its input
    p2 = synth.make_problem("int4", 16, N, N, seed=79)
    pre2 = prepack_dev(p2)
    torch.cuda.synchronize()
    outs2 = []
    for A, pre in zip(As, pres):
        outs2.append(wq.gemm_prepacked(A, pre, inputs_ready=True))
    y = wq.gemm_prepacked(outs2[-1], pre2, overlap=True)
    total = sum(o.float().sum() for o in outs2)   # a plain stream consumer of every output
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    for p, o, o2 in zip(ps, outs, outs2):
        Ce, S = oracle_ref(p)
        assert_parity(o.float().cpu().numpy().astype(np.float64), Ce, S, "bf16", "ready chain")
        assert torch.equal(o, o2)
    a_bits = outs2[-1].view(torch.int16).cpu().numpy().view(np.uint16)
    Ce, S = oracle_ref(dict(p2, A=a_bits))
    assert_parity(y.float().cpu().numpy().astype(np.float64), Ce, S, "bf16", "dependent after ready chain")
    assert float(total) == float(sum(o.float().sum() for o in outs2))


def test_overlapped_launches_chain_correctly():
    """Chained calls with WQ_LAUNCH_OVERLAP, each reading the previous call's
    output as its activations."""
    K = N = 1024
    ps = [synth.make_problem("int4", 4, N, K, seed=50 + i) for i in range(3)]
    pres = [prepack_dev(p) for p in ps]
    x = torch.from_numpy(ps[0]["A"].view(np.int16)).view(torch.bfloat16).cuda()
    outs = []
    for pre in pres:
        x = wq.gemm_prepacked(x, pre, overlap=True)
        outs.append(x)
    torch.cuda.synchronize()
    a_bits = ps[0]["A"]
    for p, o in zip(ps, outs):
        Ce, S = oracle_ref(dict(p, A=a_bits))
        assert_parity(o.float().cpu().numpy().astype(np.float64), Ce, S, "bf16", "prepacked overlap chain")
        a_bits = o.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("M,K", [(16, 8192), (16, 16384), (5, 16384), (1, 16384)])
def test_long_rows(M, K, kernel):
    """K up to the kernel's limit; 16 activation rows of K = 8192 do not fit
    beside the weights, so the call takes CTAs of fewer rows."""
    p = synth.make_problem("int4", M, 96, K, seed=K + M)
    check_pre(p, "fp32", what=f"{kernel} K={K} M={M}", ready=ready_for(kernel))


def test_k_above_limit_is_unsupported():
    p = synth.make_problem("nvfp4", 1, 16, 16384 + 128, seed=1)
    pre = prepack_dev(p)
    A, _, _, _ = to_dev(p)
    with pytest.raises(wq.WQError) as e:
        wq.gemm_prepacked(A, pre)
    assert e.value.status == wq.WQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("fmt", ["int4", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M", [1, 16, 40])
def test_fused_epilogue(fmt, M, kernel):
    p = synth.make_problem(fmt, M, 256, 1024, seed=M + 3)
    rng = np.random.default_rng(M)
    bias = synth.bf16_bits((rng.normal(size=256) * 0.5).astype(np.float32))
    res = synth.bf16_bits(rng.normal(size=(M, 128)).astype(np.float32))
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    out = "fp32" if M % 2 else "bf16"
    Y = run_pre(p, out, bias=dev(bias), residual=dev(res), gated=True, ready=ready_for(kernel))
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    Ye, T = oracle.epilogue(C, S, bias, res, True, out)
    assert not (np.abs(Y - Ye) > T).any()


@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_workload_full_size(M, kernel):
    """The decode configuration (int4 g128, N = 8192, K = 3072, bf16 out) in
    the launch configurations the bench times (the ring kernel with its
    inputs ready, the staged kernel overlapped): oracle on sampled columns
    (all rows)."""
    p = synth.workload_problem("decode_int4", M=M, seed=3)
    C = run_pre(p, "bf16", overlap=True, ready=ready_for(kernel))
    cols = sample(p["N"], 96, M)
    Ce, S = oracle_ref(p, cols=cols)
    assert_parity(C[:, cols], Ce, S, "bf16", f"decode M={M}")


def test_side_stream_and_guard_region():
    p = synth.make_problem("nvfp4", 12, 72, 256, seed=10)
    A, packed, scales, zeros = to_dev(p)
    s = torch.cuda.Stream()
    buf = torch.full((12 * 72 + 256,), 3.0, device="cuda")
    with torch.cuda.stream(s):
        pre = wq.prepack(packed, scales, zeros, "nvfp4")
        wq.gemm_prepacked(A, pre, out_dtype="fp32", out=buf[: 12 * 72].view(12, 72))
    s.synchronize()
    assert torch.all(buf[12 * 72:] == 3.0)
    Ce, S = oracle_ref(p)
    assert_parity(buf[: 12 * 72].view(12, 72).cpu().numpy().astype(np.float64), Ce, S, "fp32", "side stream")


# -- the tensor-core kernel on prepacked weights (M > 16) ---------------------------
def run_tc(p, out="fp32", workspace=None, **epi):
    A, _, _, _ = to_dev(p)
    pre = prepack_dev(p)
    C = wq.gemm_prepacked(A, pre, out_dtype=out, path="tc", workspace=workspace, **epi)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    return C.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("fmt,N,K", [("int4", 256, 1024), ("int4", 200, 640), ("nvfp4", 256, 1024),
                                     ("nvfp4", 136, 576), ("mxfp4", 256, 1024), ("mxfp4", 72, 320)])
@pytest.mark.parametrize("M", [17, 96, 300])
def test_tc_parity(fmt, N, K, M):
    """Ragged N (row blocks past N read as zero by the tensor map), K with a
    half-empty last 128-k block (fp4), several M tiles."""
    p = synth.make_problem(fmt, M, N, K, seed=M + N)
    C = run_tc(p, "fp32" if M % 2 else "bf16")
    Ce, S = oracle_ref(p)
    assert_parity(C, Ce, S, "fp32" if M % 2 else "bf16", f"tc {fmt} M={M} N={N} K={K}")


@pytest.mark.parametrize("fmt", ["int4", "nvfp4", "mxfp4"])
def test_tc_streamk_workspace(fmt, monkeypatch):
    """A shape whose whole tiles fill the SMs badly runs split (stream-K) with a
    workspace; same parity, and the workspace's flag words are left zero."""
    monkeypatch.setenv("WQ_TC_CSK", "0")   # stream-K, not the cluster split of these few tiles
    M, N, K = 128, 3072, 3072
    p = synth.make_problem(fmt, M, N, K, seed=5)
    ws = wq.workspace(M, N, K, fmt, p["group"], torch.device("cuda:0"))
    assert ws is not None
    C = run_tc(p, "bf16", workspace=ws)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert int(ws[:sms * 4].count_nonzero()) == 0
    cols = sample(N, 64, 1)
    Ce, S = oracle_ref(p, cols=cols)
    assert_parity(C[:, cols], Ce, S, "bf16", f"tc stream-K {fmt}")


@pytest.mark.parametrize("M", [40, 200])
def test_tc_second_decode_steps(M):
    p = synth.make_problem("int4", M, 144, 1024, seed=M + 1)
    rng = np.random.default_rng(M)
    z = p["zeros"].copy()
    big = rng.random(z.shape) < 0.3
    z[big] = rng.integers(129, 256, size=int(big.sum()), dtype=np.uint8)
    p["zeros"] = z
    C = run_tc(p)
    Ce, S = oracle_ref(p)
    assert_parity(C, Ce, S, "fp32", f"tc int4 big zeros M={M}")
    q = synth.make_problem("mxfp4", M, 144, 1024, seed=M + 2)
    E = q["scales"].copy()
    big = rng.random(E.shape) < 0.3
    E[big] = rng.integers(143, 161, size=int(big.sum()), dtype=np.uint8)
    q["scales"] = E
    C = run_tc(q)
    Ce, S = oracle_ref(q)
    assert_parity(C, Ce, S, "fp32", f"tc mxfp4 E>142 M={M}")


def test_tc_one_hot_selects_weight():
    N, K = 128, 512
    p = synth.make_problem("int4", 32, N, K, seed=12)
    ks = np.arange(32) * 16 + (np.arange(32) % 16)
    A = np.zeros((32, K), np.float32)
    A[np.arange(32), ks] = 1.0
    p["A"] = synth.bf16_bits(A)
    W64, _ = oracle.dequant(p["packed"], p["scales"], p["zeros"], "int4", 128)
    assert np.array_equal(run_tc(p), W64[:, ks].T)


def test_tc_fused_epilogue():
    M = 130
    p = synth.make_problem("nvfp4", M, 256, 1024, seed=77)
    rng = np.random.default_rng(M)
    bias = synth.bf16_bits((rng.normal(size=256) * 0.5).astype(np.float32))
    res = synth.bf16_bits(rng.normal(size=(M, 128)).astype(np.float32))
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    Y = run_tc(p, "bf16", bias=dev(bias), residual=dev(res), gated=True)
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], "nvfp4", 16)
    Ye, T = oracle.epilogue(C, S, bias, res, True, "bf16")
    assert not (np.abs(Y - Ye) > T).any()


def test_tc_large_nvfp4_prepacked():
    """The bench's own large-M instance: 8192^3 NVFP4 through
    gemm_prepacked(A, prepack(...)) with the default plan (tiles of 256 rows
    on persistent CTAs, the plain instance).  64 random rows (all 8192
    columns) and 64 random columns (all 8192 rows), plus the first and last
    of each, against the oracle on the original weight."""
    p = synth.workload_problem("large_nvfp4")
    A, _, _, _ = to_dev(p)
    pre = prepack_dev(p)
    C = wq.gemm_prepacked(A, pre)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    rows, cols = sample(8192, 64, 0), sample(8192, 64, 1)
    Cr, Cc = host_rows_cols(C, rows, cols)
    del C, A, pre
    Ce, S = oracle_ref(p, rows=rows)
    assert_parity(Cr, Ce, S, "bf16", "large_nvfp4 prepacked rows")
    Ce, S = oracle_ref(p, cols=cols)
    assert_parity(Cc, Ce, S, "bf16", "large_nvfp4 prepacked cols")


def test_tc_prefill_workload_full_size():
    """The prefill configuration (MXFP4, M = 2048, N = K = 3072, bf16 out) on
    prepacked weights: oracle on sampled rows and columns."""
    p = synth.workload_problem("prefill_mxfp4", seed=2)
    A, _, _, _ = to_dev(p)
    pre = prepack_dev(p)
    C = wq.gemm_prepacked(A, pre).float().cpu().numpy().astype(np.float64)
    assert wq.wq_get_device_error() == wq.WQ_OK
    rows, cols = sample(p["M"], 24, 0), sample(p["N"], 24, 1)
    Ce, S = oracle_ref(p, rows=rows)
    assert_parity(C[rows], Ce, S, "bf16", "prefill rows")
    Ce, S = oracle_ref(p, cols=cols)
    assert_parity(C[:, cols], Ce, S, "bf16", "prefill cols")


def test_auto_route_matches_both_kernels():
    """AUTO sends M > 16 to the tensor-core kernel; the small-M kernel (forced
    GEMV path) gives a result within the same gate."""
    p = synth.make_problem("int4", 48, 256, 1024, seed=3)
    A, _, _, _ = to_dev(p)
    pre = prepack_dev(p)
    Ce, S = oracle_ref(p)
    for path in ("auto", "gemv", "tc"):
        C = wq.gemm_prepacked(A, pre, out_dtype="fp32", path=path).cpu().numpy().astype(np.float64)
        assert_parity(C, Ce, S, "fp32", f"route {path}")


@pytest.mark.parametrize("layer", list(synth.LAYER_SHAPES))
@pytest.mark.parametrize("M", [1, 16, 128, 2048])
def test_layer_sweep_prepacked(layer, M):
    """Every decoder projection on prepacked weights at every M, the tied LM
    head (128256 rows, 8016 row blocks over the SMs; its prepacked buffer is
    207 MB, its M = 2048 output 0.5 GB) included: oracle on sampled rows and
    columns, copied from the device alone, the calls chained as in decode."""
    p = synth.layer_problem(layer, M)
    A, _, _, _ = to_dev(p)
    pre = prepack_dev(p)
    C = wq.gemm_prepacked(A, pre, overlap=True)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    rows, cols = sample(p["M"], 8, 0), sample(p["N"], 48, 1)
    Cr, Cc = host_rows_cols(C, rows, cols)
    del C, pre
    Ce, S = oracle_ref(p, rows=rows)
    assert_parity(Cr, Ce, S, "bf16", f"{layer} M={M} rows")
    Ce, S = oracle_ref(p, cols=cols)
    assert_parity(Cc, Ce, S, "bf16", f"{layer} M={M} cols")


@pytest.mark.parametrize("fmt,M,N", [("int4", 128, 128256), ("int4", 256, 8192), ("nvfp4", 128, 128256)])
def test_tc_repeated_calls_bit_identical(fmt, M, N):
    """The tensor-core kernel is deterministic: every k-step's stage copy is
    decoded only after it landed, whatever order the copies complete in, so
    200 repeats of the same call give the same bits (the first checked
    against the oracle on sampled rows).  The output block is poisoned with
    NaN before each call, so a store that never happens shows too."""
    K = 3072
    p = synth.make_problem(fmt, M, N, K, seed=11)
    A, _, _, _ = to_dev(p)
    pre = prepack_dev(p)
    first = wq.gemm_prepacked(A, pre, path="tc")
    torch.cuda.synchronize()
    rows = sample(M, 6, 2)
    Ce, S = oracle_ref(p, rows=rows)
    assert_parity(first.float().cpu().numpy().astype(np.float64)[rows], Ce, S, "bf16", f"{fmt} M={M} N={N}")
    ref = first.view(torch.int16).clone()
    del first
    differing = []
    for r in range(200):
        torch.full((M, N), float("nan"), device=A.device, dtype=torch.bfloat16)   # freed at once: the next block
        C = wq.gemm_prepacked(A, pre, path="tc")
        n_diff = int((C.view(torch.int16) != ref).sum())
        if n_diff:
            differing.append((r, n_diff))
        del C
    assert wq.wq_get_device_error() == wq.WQ_OK
    assert not differing, f"{len(differing)}/200 repeats differ from the first (repeat, elements): {differing[:8]}"


# -- fp4 tiles of more than 256 activation rows: two MMAs on one decode -------------
@pytest.mark.parametrize("bm", [288, 320, 352, 384])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("layout", ["plain", "prepacked"])
def test_tc_two_mma_tiles(fmt, bm, layout, monkeypatch):
    """Tile heights above one MMA's 256 rows (forced): the second MMA's
    activation box is ragged (M = bm - 40), wholly past M (M = bm / 2 - 8),
    or the start of a second, ragged m-tile (M = 2 bm - 8).  N spans three
    weight tiles, the last ragged; K nine k-steps."""
    monkeypatch.setenv("WQ_TC_BM", str(bm))
    for M in (bm - 40, bm // 2 - 8, 2 * bm - 8):
        p = synth.make_problem(fmt, M, 300, 576, seed=bm + M)
        if layout == "prepacked":
            C = run_tc(p, "fp32")
        else:
            from gpu_util import gpu_gemm
            C = gpu_gemm(p, "fp32", path="tc")
        Ce, S = oracle_ref(p)
        assert_parity(C, Ce, S, "fp32", f"{fmt} bm={bm} M={M} {layout}")


def test_tc_two_mma_tiles_fused_epilogue(monkeypatch):
    """The fused epilogue (bias, SiLU-gated pairs, residual) on a 320-row tile."""
    monkeypatch.setenv("WQ_TC_BM", "320")
    M = 600
    p = synth.make_problem("nvfp4", M, 256, 1024, seed=78)
    rng = np.random.default_rng(M)
    bias = synth.bf16_bits((rng.normal(size=256) * 0.5).astype(np.float32))
    res = synth.bf16_bits(rng.normal(size=(M, 128)).astype(np.float32))
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    Y = run_tc(p, "bf16", bias=dev(bias), residual=dev(res), gated=True)
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], "nvfp4", 16)
    Ye, T = oracle.epilogue(C, S, bias, res, True, "bf16")
    assert not (np.abs(Y - Ye) > T).any()


def test_tc_int4_keeps_256_rows(monkeypatch):
    """int4 tiles stay within one MMA (its hi and lo weight buffers take the
    TMEM columns a second accumulator half would need): a forced height
    above 256 falls back to the default choice and the result holds."""
    monkeypatch.setenv("WQ_TC_BM", "320")
    p = synth.make_problem("int4", 400, 256, 1024, seed=79)
    C = run_tc(p, "fp32")
    Ce, S = oracle_ref(p)
    assert_parity(C, Ce, S, "fp32", "int4 forced 320")
