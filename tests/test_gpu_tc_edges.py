"""Edge combinations of the tensor-core kernel's newer paths, each against
the oracle: the decode look-ahead across segment boundaries of every kind
(whole tiles, stream-K segments of odd lengths, several per CTA), cluster
split-K with fp32 output and a gated epilogue together, and the bulk store
over the stage ring with ragged M and N."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import check_full, check_sampled, gpu_gemm_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["int4", "nvfp4"])
@pytest.mark.parametrize("ctas", ["13", "37", "150"])
def test_lookahead_over_streamk_segments(fmt, ctas, monkeypatch):
    """Stream-K with CTA counts that cut tiles at odd k-steps: each CTA walks
    a partial segment then whole ones, and decodes each next segment's first
    k-step ahead."""
    monkeypatch.setenv("WQ_TC_CSK", "0")
    monkeypatch.setenv("WQ_TC_STREAMK", "1")
    monkeypatch.setenv("WQ_TC_SK_G", ctas)
    group = 64 if fmt == "int4" else None   # K = 2112 is not a multiple of 128
    p = synth.make_problem(fmt, 300, 1000, 2112, group=group, seed=int(ctas))   # 33 k-steps per tile
    n = wq.wq_gemm_workspace_size(300, 1000, 2112, wq.FORMATS[fmt], p["group"])
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    check_full(p, "fp32", path="tc", workspace=ws, what=f"{fmt} stream-K G={ctas}")


@pytest.mark.parametrize("M", [700, 1500])
def test_lookahead_over_whole_tiles(M, monkeypatch):
    """Whole tiles, several per CTA (forced 32-row tiles), ragged M and N."""
    monkeypatch.setenv("WQ_TC_CSK", "0")
    monkeypatch.setenv("WQ_TC_BM", "32")
    p = synth.make_problem("mxfp4", M, 1160, 640, seed=M)
    check_sampled(p, "bf16", k=24, path="tc", what=f"M={M} 32-row tiles")


def test_cluster_split_fp32_gated_epilogue(monkeypatch):
    monkeypatch.setenv("WQ_TC_CSK", "1")
    p = synth.make_problem("int4", 90, 640, 3072, seed=5)
    rng = np.random.default_rng(5)
    bias = synth.bf16_bits((rng.normal(size=640) * 0.5).astype(np.float32))
    res = synth.bf16_bits(rng.normal(size=(90, 320)).astype(np.float32))
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    A, packed, scales, zeros = to_dev(p)
    Y = wq.gemm(A, packed, scales, zeros, "int4", out_dtype="fp32", path="tc", bias=dev(bias), residual=dev(res),
                gated=True)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], "int4", 128)
    Ye, T = oracle.epilogue(C, S, bias, res, True, "fp32")
    err = np.abs(Y.cpu().numpy().astype(np.float64) - Ye)
    assert (err <= T).all(), float(np.max(err - T))


def test_bulk_store_over_the_ring_ragged(monkeypatch):
    """352-row two-MMA tiles, one per CTA, with M and N not multiples of the
    tile: the tensor map clips both boxes."""
    monkeypatch.setenv("WQ_TC_CSK", "0")
    monkeypatch.setenv("WQ_TC_BM", "352")
    p = synth.make_problem("nvfp4", 1000, 1544, 512, seed=9)   # 3 x 13 = 39 tiles
    C1 = gpu_gemm_dev(p, "bf16", path="tc")
    monkeypatch.setenv("WQ_TC_NO_TMA_STORE", "1")
    C2 = gpu_gemm_dev(p, "bf16", path="tc")
    assert torch.equal(C1, C2)
    monkeypatch.delenv("WQ_TC_NO_TMA_STORE")
    check_sampled(p, "bf16", k=24, path="tc", what="352-row tiles, ragged")
