"""Programmatic dependent launch on the tensor-core path (WQ_LAUNCH_OVERLAP,
or WQ_LAUNCH_INPUTS_READY, which this path treats the same way): a call may
start while its predecessor runs, reads A only after the predecessor has
completed, and writes C (and stream-K partials) only after that.  Checked
on chains where the order matters -- a call reading its predecessor's
output (read after write) and a call overwriting its predecessor's input
(write after read) -- under every tile plan."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import assert_parity, to_dev

pytestmark = pytest.mark.gpu

PLANS = {"auto": {}, "whole": {"WQ_TC_CSK": "0"}, "streamk": {"WQ_TC_CSK": "0", "ws": True},
         "thread-stores": {"WQ_TC_CSK": "0", "WQ_TC_NO_TMA_STORE": "1"}}


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run(A, pw, fmt, out, flag, ws):
    A_, packed, scales, zeros = A, *pw
    return wq.gemm(A_, packed, scales, zeros, fmt, out=out, path="tc", workspace=ws, overlap=flag == "overlap",
                   inputs_ready=flag == "ready")


@pytest.mark.parametrize("plan", list(PLANS))
@pytest.mark.parametrize("flag", ["overlap", "ready"])
def test_read_after_write(plan, flag, monkeypatch):
    """C1 = A . W1^T, then C2 = C1 . W2^T chained: the second call must read
    the first one's finished output."""
    for k, v in PLANS[plan].items():
        if k != "ws":
            monkeypatch.setenv(k, v)
    M, N1, K1, N2 = 256, 1024, 512, 640
    p1 = synth.make_problem("int4", M, N1, K1, seed=1)
    p2 = synth.make_problem("nvfp4", M, N2, N1, seed=2)
    A1, *w1 = to_dev(p1)
    _, *w2 = to_dev(p2)
    ws = None
    if "ws" in PLANS[plan]:
        n = max(wq.wq_gemm_workspace_size(M, N1, K1, wq.WQ_INT4, 128),
                wq.wq_gemm_workspace_size(M, N2, N1, wq.WQ_NVFP4, 16))
        ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    C1 = torch.empty(M, N1, dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty(M, N2, dtype=torch.bfloat16, device="cuda")
    for rep in range(3):
        C1.fill_(float("nan"))   # a read before the write would see NaN
        torch.cuda.synchronize()
        run(A1, w1, "int4", C1, flag, ws)
        run(C1, w2, "nvfp4", C2, flag, ws)
        torch.cuda.synchronize()
        assert wq.wq_get_device_error() == wq.WQ_OK
    a2 = bits(C1)
    Ce, S = oracle.gemm(a2, p2["packed"], p2["scales"], p2["zeros"], "nvfp4", 16)
    assert_parity(C2.float().cpu().numpy().astype(np.float64), Ce, S, "bf16", f"RAW {plan} {flag}")


@pytest.mark.parametrize("plan", list(PLANS))
def test_write_after_read(plan, monkeypatch):
    """A long call reads X; the next call, chained, writes its C into X: the
    first call must have read all of X before the second one's stores."""
    for k, v in PLANS[plan].items():
        if k != "ws":
            monkeypatch.setenv(k, v)
    M, N, K = 2048, 3072, 3072
    p1 = synth.make_problem("int4", M, N, K, seed=3)
    p2 = synth.make_problem("int4", M, K, 256, seed=4)   # writes an (M, K) result: X's shape
    X, *w1 = to_dev(p1)
    A2, *w2 = to_dev(p2)
    ws = None
    if "ws" in PLANS[plan]:
        n = max(wq.wq_gemm_workspace_size(M, N, K, wq.WQ_INT4, 128), wq.wq_gemm_workspace_size(M, K, 256, wq.WQ_INT4, 128))
        ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    C1 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    run(X, w1, "int4", C1, "overlap", ws)
    run(A2, w2, "int4", X, "overlap", ws)   # overwrites X
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    rows = np.array([0, 1, 777, 2047])
    Ce, S = oracle.gemm(p1["A"], p1["packed"], p1["scales"], p1["zeros"], "int4", 128, rows=rows)
    assert_parity(C1[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64), Ce, S, "bf16",
                  f"WAR {plan}")
