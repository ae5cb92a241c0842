"""The small-M kernels' final stores: plain output in 16-byte pieces
where C is 16-byte aligned and N a multiple of 8 (bf16) or 4 (fp32), else
one output per thread.  Parity against the oracle, and the same bits as the
one-output stores (WQ_GEMV_SCALAR_STORE), on both kernels (the ring kernel
for calls whose inputs are ready, the staged kernel for the others): ragged
row blocks (N not a multiple of 16), one and two tiles of activation rows,
several 16-row chunks, and the rows that keep the one-output stores."""
import numpy as np
import pytest
import torch

import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import assert_parity, gpu_gemm_dev, oracle_ref, to_dev

pytestmark = pytest.mark.gpu


def run(p, out, ready, monkeypatch, scalar):
    if scalar:
        monkeypatch.setenv("WQ_GEMV_SCALAR_STORE", "1")
    else:
        monkeypatch.delenv("WQ_GEMV_SCALAR_STORE", raising=False)
    A, packed, scales, zeros = to_dev(p)
    pre = wq.prepack(packed, scales, zeros, p["fmt"], p["group"])
    C = wq.gemm_prepacked(A, pre, out_dtype=out, inputs_ready=ready)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    return C


@pytest.mark.parametrize("kernel", ["ring", "staged"])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("fmt,M,N,K", [
    ("int4", 16, 1000, 512),     # 62.5 row blocks: the last one half full
    ("int4", 3, 264, 384),
    ("int4", 20, 520, 256),      # two 16-row chunks, the second of 4 rows
    ("nvfp4", 9, 1000, 512),
    ("mxfp4", 1, 2056, 1024),
])
def test_pieces_same_bits_as_single_stores(kernel, out, fmt, M, N, K, monkeypatch):
    monkeypatch.setenv("WQ_GEMV_PRE_KERNEL", kernel)
    p = synth.make_problem(fmt, M, N, K, seed=M * 7 + N)
    ready = kernel == "ring"
    C1 = run(p, out, ready, monkeypatch, scalar=False)
    C2 = run(p, out, ready, monkeypatch, scalar=True)
    assert torch.equal(C1, C2), f"{kernel} {out} {fmt} {M}x{N}x{K}"
    Ce, S = oracle_ref(p)
    assert_parity(C1.float().cpu().numpy().astype(np.float64), Ce, S, out, f"{kernel} {out} {fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("kernel", ["ring", "staged"])
@pytest.mark.parametrize("out,N", [("bf16", 1004), ("fp32", 1002)])
def test_unaligned_rows_keep_single_stores(kernel, out, N, monkeypatch):
    """Rows whose bytes are not a multiple of 16 (C itself is 16-byte aligned
    by the interface) take the one-output stores: within the gate, and the
    same bits with the pieces switched off."""
    monkeypatch.setenv("WQ_GEMV_PRE_KERNEL", kernel)
    p = synth.make_problem("int4", 16, N, 512, seed=N)
    ready = kernel == "ring"
    Ce, S = oracle_ref(p)
    C1 = run(p, out, ready, monkeypatch, scalar=False)
    C2 = run(p, out, ready, monkeypatch, scalar=True)
    assert torch.equal(C1, C2)
    assert_parity(C1.float().cpu().numpy().astype(np.float64), Ce, S, out, f"{kernel} {out} N={N}")


def test_ready_calls_into_one_output_keep_stream_order(monkeypatch):
    """Calls with their inputs declared ready compute before the preceding
    call completes and store after it: consecutive calls into the same C
    leave the last call's result, and a plain consumer between them sees
    the earlier one."""
    monkeypatch.delenv("WQ_GEMV_SCALAR_STORE", raising=False)
    monkeypatch.setenv("WQ_GEMV_PRE_KERNEL", "ring")
    N, K = 2048, 3072
    ps = [synth.make_problem("int4", M, N, K, seed=90 + i) for i, M in enumerate((16, 16, 16, 16))]
    pres = []
    for p in ps:
        _, packed, scales, zeros = to_dev(p)
        pres.append(wq.prepack(packed, scales, zeros, p["fmt"], p["group"]))
    A = to_dev(ps[0])[0]
    torch.cuda.synchronize()
    C = torch.empty((16, N), dtype=torch.bfloat16, device="cuda")
    snaps = []
    for rep in range(3):
        for i, pre in enumerate(pres):
            wq.gemm_prepacked(A, pre, out=C, inputs_ready=True)
            if i == 1:
                snaps.append(C.clone())   # a plain stream consumer after the second call
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    A_bits = ps[0]["A"]
    for idx, got in ((3, C), (1, snaps[-1])):
        Ce, S = oracle_ref(dict(ps[idx], A=A_bits))
        assert_parity(got.float().cpu().numpy().astype(np.float64), Ce, S, "bf16", f"call {idx} into a shared C")
    assert all(torch.equal(snaps[0], s) for s in snaps[1:])


@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("fmt,M,N,K", [("int4", 16, 1000, 512), ("int4", 4, 8192, 3072), ("nvfp4", 1, 264, 256),
                                       ("mxfp4", 12, 520, 1024), ("int4", 16, 1004, 512)])
def test_input_layout_pieces_same_bits(out, fmt, M, N, K, monkeypatch):
    """The input-layout streaming kernel (wq_gemm at M <= 16) stores the same
    bits in pieces as one output at a time, within the gate."""
    p = synth.make_problem(fmt, M, N, K, seed=M + N + K)
    monkeypatch.delenv("WQ_GEMV_SCALAR_STORE", raising=False)
    C1 = gpu_gemm_dev(p, out)
    monkeypatch.setenv("WQ_GEMV_SCALAR_STORE", "1")
    C2 = gpu_gemm_dev(p, out)
    assert torch.equal(C1, C2), f"{out} {fmt} {M}x{N}x{K}"
    Ce, S = oracle_ref(p)
    assert_parity(C1.float().cpu().numpy().astype(np.float64), Ce, S, out, f"input layout {out} {fmt} {M}x{N}x{K}")
