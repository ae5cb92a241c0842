"""wq_gemm_static: the tensor-core path's tile splitting with the library's
own scratch (a fixed device array found once per device) -- no allocation by
the caller or the library.  Parity against the oracle, the scratch left
usable across calls, and the refusal of a shape whose split would need more
scratch than is there."""
import ctypes

import numpy as np
import pytest
import torch

import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import assert_parity, oracle_ref, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def streamk_not_clusters(monkeypatch):
    """The split shapes have few tiles, which the library would otherwise split
    over thread-block clusters (tests/test_gpu_cluster.py) instead."""
    monkeypatch.setenv("WQ_TC_CSK", "0")


def run_static(p, out="fp32", path=wq.WQ_PATH_AUTO):
    A, packed, scales, zeros = to_dev(p)
    odt = torch.float32 if out == "fp32" else torch.bfloat16
    C = torch.empty((p["M"], p["N"]), dtype=odt, device="cuda")
    fmt = wq.FORMATS[p["fmt"]] | (wq.WQ_OUT_F32 if out == "fp32" else 0)
    st = wq.wq_gemm_static(A.data_ptr(), packed.data_ptr(), scales.data_ptr(),
                           zeros.data_ptr() if zeros is not None else None, C.data_ptr(),
                           p["M"], p["N"], p["K"], fmt, p["group"],
                           torch.cuda.current_stream().cuda_stream, path)
    torch.cuda.synchronize()
    return st, C.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("fmt,M,N,K", [("int4", 128, 3072, 3072), ("nvfp4", 17, 384, 4096),
                                       ("mxfp4", 300, 1000, 1024), ("int4", 4, 512, 1024)])
def test_static_scratch_parity(fmt, M, N, K):
    p = synth.make_problem(fmt, M, N, K, seed=M + K)
    # the split really happens for the tensor-core shapes
    if M > 16:
        assert wq.wq_gemm_workspace_size(M, N, K, wq.FORMATS[fmt], p["group"]) > 0
    for rep in range(2):   # the second call finds the flags the first left zero
        st, C = run_static(p)
        assert st == wq.WQ_OK
        assert wq.wq_get_device_error() == wq.WQ_OK
        Ce, S = oracle_ref(p)
        assert_parity(C, Ce, S, "fp32", f"static {fmt} {M}x{N}x{K} call {rep}")


def test_static_scratch_refuses_oversize(monkeypatch):
    p = synth.make_problem("int4", 128, 3072, 3072, seed=2)
    need = wq.wq_gemm_workspace_size(128, 3072, 3072, wq.WQ_INT4, 128)
    monkeypatch.setenv("WQ_STATIC_WS_CAP", str(need - 1))
    st, _ = run_static(p)
    assert st == wq.WQ_ERR_UNSUPPORTED
    monkeypatch.setenv("WQ_STATIC_WS_CAP", str(need))
    st, C = run_static(p)
    assert st == wq.WQ_OK
    Ce, S = oracle_ref(p)
    assert_parity(C, Ce, S, "fp32", "static at exact capacity")


def test_static_call_allocates_no_device_memory():
    """The entry point's defining property: after a first call (which finds
    the scratch's address), further calls that split tiles over the SMs
    leave the device's free memory unchanged -- neither the caller nor the
    library allocated anything."""
    p = synth.make_problem("int4", 128, 3072, 3072, seed=4)
    assert wq.wq_gemm_workspace_size(128, 3072, 3072, wq.WQ_INT4, 128) > 0
    A, packed, scales, zeros = to_dev(p)
    C = torch.empty((128, 3072), dtype=torch.float32, device="cuda")
    h = torch.cuda.current_stream().cuda_stream

    def call():
        return wq.wq_gemm_static(A.data_ptr(), packed.data_ptr(), scales.data_ptr(), zeros.data_ptr(),
                                 C.data_ptr(), 128, 3072, 3072, wq.WQ_INT4 | wq.WQ_OUT_F32, 128, h,
                                 wq.WQ_PATH_AUTO)

    assert call() == wq.WQ_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert call() == wq.WQ_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    Ce, S = oracle_ref(p)
    assert_parity(C.cpu().numpy().astype(np.float64), Ce, S, "fp32", "static, no allocation")


def test_static_scratch_after_a_timeout(monkeypatch):
    """A call whose stream-K wait gave up (WQ_TC_FLAG_WAIT_NS=0) leaves flags
    set in the library's scratch.  Once wq_get_device_error() has reported
    the timeout, the next call clears the scratch's flag words on its stream
    before its kernel runs, so it reads no partial sum of the failed call."""
    bad = synth.make_problem("int4", 128, 3072, 3072, seed=40)
    good = synth.make_problem("int4", 128, 3072, 3072, seed=41)
    assert wq.wq_get_device_error() == wq.WQ_OK
    monkeypatch.setenv("WQ_TC_FLAG_WAIT_NS", "0")
    st, _ = run_static(bad)
    assert st == wq.WQ_OK
    assert wq.wq_get_device_error() == wq.WQ_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("WQ_TC_FLAG_WAIT_NS")
    Ce, S = oracle_ref(good)
    for rep in range(2):
        st, C = run_static(good)
        assert st == wq.WQ_OK
        assert wq.wq_get_device_error() == wq.WQ_OK
        assert_parity(C, Ce, S, "fp32", f"static after a timeout, call {rep}")


def test_static_checks_the_description_first():
    """Format and path are validated before the scratch; the scratch size
    only limits calls that take the tensor-core path."""
    FAKE = 1 << 20
    assert wq.wq_gemm_static(FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 7, 16, None, 0) == wq.WQ_ERR_INVALID_ARG
    assert wq.wq_gemm_static(FAKE, FAKE, FAKE, None, FAKE, 4, 8, 64, 0, 16, None, 9) == wq.WQ_ERR_INVALID_ARG


def test_static_gemv_path_ignores_the_scratch_cap(monkeypatch):
    """A call that runs on the small-M kernel uses no scratch, so even a
    zero usable scratch does not refuse it."""
    monkeypatch.setenv("WQ_STATIC_WS_CAP", "0")
    p = synth.make_problem("int4", 128, 256, 1024, seed=6)
    st, C = run_static(p, path=wq.WQ_PATH_GEMV)
    assert st == wq.WQ_OK
    Ce, S = oracle_ref(p)
    assert_parity(C, Ce, S, "fp32", "static, GEMV path, no scratch")


def test_static_cluster_split_needs_no_scratch(monkeypatch):
    """Few tiles split over thread-block clusters add their partial sums on
    chip: the call uses no scratch, so even a zero usable scratch serves it."""
    monkeypatch.setenv("WQ_TC_CSK", "1")
    monkeypatch.setenv("WQ_STATIC_WS_CAP", "0")
    p = synth.make_problem("int4", 128, 3072, 3072, seed=8)
    assert wq.wq_gemm_workspace_size(128, 3072, 3072, wq.WQ_INT4, 128) == 0
    st, C = run_static(p)
    assert st == wq.WQ_OK
    assert wq.wq_get_device_error() == wq.WQ_OK
    Ce, S = oracle_ref(p)
    assert_parity(C, Ce, S, "fp32", "static, cluster split-K")
