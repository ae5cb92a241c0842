"""The tensor-core path with a workspace (wq_gemm_ws): tiles whose k-steps
are shared by several CTAs are finished by the CTA holding the last k-step,
from the partial sums the others leave in the workspace.  Parity against the
oracle on the workloads, on shapes that split tiles over many CTAs, and the
workspace contract (zero before first use, left zero by every call)."""
import numpy as np
import pytest
import torch

import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import check_full, check_sampled, gpu_gemm, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def streamk_not_clusters(monkeypatch):
    """These shapes have few tiles, which the library would otherwise split
    over thread-block clusters (tests/test_gpu_cluster.py) instead."""
    monkeypatch.setenv("WQ_TC_CSK", "0")


def ws_for(p):
    n = wq.wq_gemm_workspace_size(p["M"], p["N"], p["K"], wq.FORMATS[p["fmt"]], p["group"])
    return torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda"), n


@pytest.mark.parametrize("force", ["0", "1"])
def test_prefill_mxfp4(force, monkeypatch):
    """The prefill workload with a workspace, both ways: whole tiles (its
    waves are 87% full, so the library keeps them whole) and split."""
    monkeypatch.setenv("WQ_TC_STREAMK", force)
    p = synth.workload_problem("prefill_mxfp4")
    ws, n = ws_for(p)
    assert (n > 0) == (force == "1")
    check_sampled(p, "bf16", workspace=ws, what=f"prefill_mxfp4 stream-K={force}")


def test_small_m_layers_split():
    """128 activation rows: 24 tiles on 152 SMs -- the library splits them."""
    p = synth.layer_problem("q", 128)
    ws, n = ws_for(p)
    assert n > 0
    check_sampled(p, "bf16", k=8, workspace=ws, what="q M=128 stream-K")


@pytest.mark.parametrize("layer", ["q", "kv", "gate_up", "down", "lm_head"])
@pytest.mark.parametrize("M", [128, 2048])
def test_layer_shapes(layer, M):
    p = synth.layer_problem(layer, M)
    ws, _ = ws_for(p)
    check_sampled(p, "bf16", k=8, workspace=ws, what=f"{layer} M={M} stream-K")


# few tiles and long K: every tile is shared by several CTAs -- as many as
# the library's CTA count gives (about tiles x sqrt(k-steps x 128 / bm)), or,
# forced, one per SM (tens of partials per tile)
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
@pytest.mark.parametrize("M,N,K", [(17, 384, 4096), (128, 128, 8192), (130, 257, 1024), (300, 1000, 4160),
                                   (64, 200, 640)])
@pytest.mark.parametrize("ctas", ["model", "all"])
def test_many_partials(fmt, M, N, K, ctas, monkeypatch):
    if ctas == "all":
        monkeypatch.setenv("WQ_TC_SK_G", "100000")   # capped at min(units, SMs)
    group = 64 if (fmt == "int4" and K % 128) else None   # K must be a multiple of the group
    p = synth.make_problem(fmt, M, N, K, group=group, seed=M + N + K)
    ws, n = ws_for(p)
    check_full(p, "fp32", path="tc", workspace=ws, what=f"{fmt} {M}x{N}x{K} stream-K")


def test_workspace_left_zero_and_reused():
    """Consecutive calls of different shapes on one workspace: each finds the
    flags it needs at zero (a stale flag would hand a consumer an old
    partial), and the flag words are zero again afterwards."""
    # a one-tile shape (a grid of a few CTAs) between shapes with larger grids
    shapes = [("int4", 128, 384, 4096), ("mxfp4", 17, 128, 8192), ("nvfp4", 300, 1000, 1024)]
    size = max(wq.wq_gemm_workspace_size(M, N, K, wq.FORMATS[f], synth.GROUP[f]) for f, M, N, K in shapes)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for f, M, N, K in shapes:
            p = synth.make_problem(f, M, N, K, seed=rep * 7 + M)
            check_full(p, "fp32", path="tc", workspace=ws, what=f"reuse {f} {M}x{N}x{K}")
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    flags = ws[:sms * 4].view(torch.int32)   # the flag words lead the workspace
    assert int(flags.abs().sum()) == 0


def test_deterministic_with_workspace():
    p = synth.make_problem("int4", 200, 640, 4096, seed=11)
    ws, _ = ws_for(p)
    C1 = gpu_gemm(p, "fp32", "tc", ws)
    C2 = gpu_gemm(p, "fp32", "tc", ws)
    assert np.array_equal(C1, C2)


def test_small_workspace_runs_whole_tiles():
    p = synth.make_problem("nvfp4", 130, 257, 2048, seed=5)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")   # below the size the shape needs
    check_full(p, "fp32", path="tc", workspace=ws, what="small workspace")


def test_ws_argument_checks():
    p = synth.make_problem("nvfp4", 40, 64, 256, seed=6)
    A, packed, scales, zeros = to_dev(p)
    C = torch.empty((40, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    args = (A.data_ptr(), packed.data_ptr(), scales.data_ptr(), None, C.data_ptr(), 40, 64, 256, 0, 16)
    assert wq.wq_gemm_ws(*args, ws.data_ptr() + 16, 1024, None, 0) == wq.WQ_ERR_ALIGN
    assert wq.wq_gemm_ws(*args, None, 1024, None, 0) == wq.WQ_ERR_INVALID_ARG
    assert wq.wq_gemm_ws(*args, None, 0, None, 0) == wq.WQ_OK
    torch.cuda.synchronize()
