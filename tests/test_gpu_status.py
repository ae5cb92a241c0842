"""The failure path of the bounded device waits, exercised without hanging or
faulting the GPU: a kernel waits on an mbarrier that nothing completes, gives
up after its wall-time bound and records WQ_ERR_DEVICE_TIMEOUT; the status is
read and cleared, and the context keeps working."""
import numpy as np
import pytest
import torch

import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import check_full

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_cleared():
    assert wq.wq_get_device_error() == wq.WQ_OK
    assert wq.wq_selftest_timeout(None) == wq.WQ_OK
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.wq_get_device_error() == wq.WQ_OK          # read clears it
    # the context is still usable: a full GEMM on both paths
    check_full(synth.make_problem("int4", 300, 256, 512, seed=1), "fp32", what="after timeout")
    check_full(synth.make_problem("nvfp4", 4, 256, 512, seed=2), "fp32", what="after timeout")
    assert wq.wq_get_device_error() == wq.WQ_OK


def test_streamk_flag_wait_runs_out(monkeypatch):
    """The real tensor-core kernel's failure path, run without a fault or a
    hang: with the stream-K flag wait bounded at 0 ns (WQ_TC_FLAG_WAIT_NS,
    read at launch) every tile owner gives up at once, raises its CTA's abort
    flag, lets the producer and the MMA issuer drain what is in flight, frees
    its tensor memory and records WQ_ERR_DEVICE_TIMEOUT; the copy and MMA
    waits keep their normal bounds.  The contributors' flags stay set, so the
    workspace must be zeroed again; then the same call is oracle-green."""
    from gpu_util import assert_parity, oracle_ref, to_dev
    M, N, K = 128, 1024, 3072            # 8 tiles on the SMs: split over many CTAs
    monkeypatch.setenv("WQ_TC_CSK", "0")   # by stream-K (the cluster split needs no flags)
    p = synth.make_problem("int4", M, N, K, seed=5)
    n = wq.wq_gemm_workspace_size(M, N, K, wq.WQ_INT4, 128)
    assert n > 0
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    A, packed, scales, zeros = to_dev(p)
    assert wq.wq_get_device_error() == wq.WQ_OK
    monkeypatch.setenv("WQ_TC_FLAG_WAIT_NS", "0")
    wq.gemm(A, packed, scales, zeros, "int4", out_dtype="fp32", workspace=ws)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.wq_get_device_error() == wq.WQ_OK
    flags = ws[: 4 * sms].view(torch.int32)
    assert int(flags.sum()) > 0            # left set by the contributors
    monkeypatch.delenv("WQ_TC_FLAG_WAIT_NS")
    ws.zero_()
    C = wq.gemm(A, packed, scales, zeros, "int4", out_dtype="fp32", workspace=ws)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    assert int(flags.sum()) == 0           # a completed call leaves them zero
    Ce, S = oracle_ref(p)
    assert_parity(C.cpu().numpy().astype(np.float64), Ce, S, "fp32", "after the flag-wait timeout")
