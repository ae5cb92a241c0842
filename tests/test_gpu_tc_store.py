"""Whole tiles of plain bf16 output on the tensor-core path: the accumulator
is staged as bf16 in shared memory and written by one bulk tensor store per
tile, which clips the rows and columns past M and N.  Parity against the
oracle on ragged shapes, the same bits as the decode warps' own stores
(WQ_TC_NO_TMA_STORE), and the shapes that keep the thread stores (fp32
output, N not a multiple of 8, a fused epilogue)."""
import numpy as np
import pytest
import torch

import weight_only_bit_w4a16_gb300 as wq
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import check_full, check_sampled, gpu_gemm_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture
def stores(monkeypatch, capfd):
    """Whole tiles (no cluster split, no workspace); returns a reader of the
    store mode of the last tensor-core call."""
    monkeypatch.setenv("WQ_TC_CSK", "0")
    monkeypatch.setenv("WQ_DEBUG", "1")
    capfd.readouterr()

    def mode():
        err = capfd.readouterr().err
        lines = [ln for ln in err.splitlines() if ln.startswith("wq: tensor-core C stores")]
        assert lines, err[-400:]
        return lines[-1].rsplit(": ", 1)[1]

    return mode


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
@pytest.mark.parametrize("M,N,K", [(300, 1000, 1024), (97, 264, 512), (520, 392, 256)])
def test_ragged_bulk_store(fmt, M, N, K, stores):
    p = synth.make_problem(fmt, M, N, K, seed=M * 3 + N)
    check_full(p, "bf16", path="tc", what=f"{fmt} {M}x{N}x{K} bulk-store epilogue")
    assert stores() == "bulk tensor"


@pytest.mark.parametrize("fmt,M,N,K,bm", [("int4", 300, 1000, 1024, 256), ("nvfp4", 2048, 3072, 3072, 128)])
def test_same_bits_as_thread_stores(fmt, M, N, K, bm, stores, monkeypatch):
    # Forced tile heights with room for the staging tile beside the ring: the
    # NVFP4 shape would take two-MMA tiles of 352 rows (thread stores, several
    # tiles per CTA), and its one-MMA tiles of 256 rows fill shared memory
    # with their six stages.
    monkeypatch.setenv("WQ_TC_BM", str(bm))
    p = synth.make_problem(fmt, M, N, K, seed=7)
    C1 = gpu_gemm_dev(p, "bf16", path="tc")
    assert stores() == "bulk tensor"
    monkeypatch.setenv("WQ_TC_NO_TMA_STORE", "1")
    C2 = gpu_gemm_dev(p, "bf16", path="tc")
    assert stores() == "threads"
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("out,N", [("fp32", 1000), ("bf16", 1001)])
def test_thread_store_shapes(out, N, stores):
    """fp32 output and rows whose bytes are not a multiple of 16 keep the
    decode warps' stores."""
    p = synth.make_problem("int4", 200, N, 512, seed=N)
    check_full(p, out, path="tc", what=f"{out} N={N}")
    assert stores() == "threads"


def test_int4_2048_bulk_store(stores):
    """int4 2048 x 3072 x 3072: tiles of at most 256 rows, staged beside the
    stage ring."""
    p = synth.make_problem("int4", 2048, 3072, 3072, seed=11)
    check_sampled(p, "bf16", k=16, path="tc", what="int4 2048x3072x3072 bulk store")
    assert stores() == "bulk tensor"


def test_prefill_two_mma_tiles_stage_over_the_ring(stores, monkeypatch):
    """The prefill workload (MXFP4 2048 x 3072 x 3072): 144 tiles of 352
    rows, one per CTA, too tall to stage beside the ring, so they stage over
    it once their MMAs are done and leave as two boxes of 176 rows; same
    bits as the decode warps' stores."""
    p = synth.workload_problem("prefill_mxfp4")
    C1 = gpu_gemm_dev(p, "bf16", path="tc")
    assert stores() == "bulk tensor"
    monkeypatch.setenv("WQ_TC_NO_TMA_STORE", "1")
    C2 = gpu_gemm_dev(p, "bf16", path="tc")
    assert stores() == "threads"
    assert torch.equal(C1, C2)
    monkeypatch.delenv("WQ_TC_NO_TMA_STORE")
    check_sampled(p, "bf16", k=16, path="tc", what="prefill bulk store over the ring")


def test_two_mma_tiles_several_per_cta_keep_thread_stores(stores, monkeypatch):
    """Tiles of 352 rows with more tiles than SMs: a CTA's ring serves its
    next tile, so these keep the decode warps' stores."""
    monkeypatch.setenv("WQ_TC_BM", "352")
    p = synth.make_problem("nvfp4", 2816, 2560, 512, seed=13)   # 8 x 20 = 160 tiles > SMs
    check_sampled(p, "bf16", k=16, path="tc", what="352-row tiles, several per CTA")
    assert stores() == "threads"
