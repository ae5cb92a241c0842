"""wq_dequant on the GPU: bit-exact against the oracle's bf16 image.

Every weight must equal the round-to-nearest-even bf16 of its exact value
(NaN compared as NaN), including every (code, scale byte) pair of the fp4
formats, every bf16 scale of int4 with every code and zero point, the
special values (NaN scales, e8m0 overflow, -0) and ragged shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from weight_only_bit_w4a16_gb300 import synth

from gpu_util import gpu_dequant_bits, to_dev

pytestmark = pytest.mark.gpu


def is_nan_bits(b):
    b = np.asarray(b, dtype=np.int64)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def assert_bits_equal(got, ref, what=""):
    nan = is_nan_bits(ref)
    assert np.array_equal(is_nan_bits(got), nan), f"{what}: NaN positions differ"
    bad = (got != ref) & ~nan
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} mismatches, first at {tuple(i)}: "
                             f"gpu={int(got[tuple(i)]):#06x} oracle={int(ref[tuple(i)]):#06x}")


def problem(fmt, N, K, packed, scales, zeros=None, group=None):
    return dict(fmt=fmt, group=group or synth.GROUP[fmt], M=0, N=N, K=K,
                A=np.zeros((0, K), np.uint16), packed=packed, scales=scales, zeros=zeros)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
@pytest.mark.parametrize("NK", [(1, 32), (3, 128), (257, 512), (1000, 3072)])
def test_dequant_random_bit_exact(fmt, NK):
    N, K = NK
    if K % synth.GROUP[fmt]:
        pytest.skip("K not a multiple of the group")
    packed, scales, zeros = synth.make_weights(fmt, N, K, seed=N + K)
    p = problem(fmt, N, K, packed, scales, zeros)
    _, ref = oracle.dequant(packed, scales, zeros, fmt, p["group"])
    assert_bits_equal(gpu_dequant_bits(p), ref, f"{fmt} {N}x{K}")


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_dequant_fp4_every_code_every_scale_byte(fmt):
    group = synth.GROUP[fmt]
    codes = np.tile(np.arange(16), 2)
    row = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    packed = np.tile(row, (256, 1))
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 32 // group, axis=1)
    p = problem(fmt, 256, 32, packed, scales)
    _, ref = oracle.dequant(packed, scales, None, fmt, group)
    assert_bits_equal(gpu_dequant_bits(p), ref, fmt)


def test_dequant_int4_every_bf16_scale_code_and_zero():
    n = np.arange(65536)
    codes = np.tile(np.arange(16), 2)
    row = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    packed = np.tile(row, (65536, 1))
    scales = n.astype(np.uint16)[:, None]
    for zeros in ((n % 16).astype(np.uint8)[:, None],          # the promised 0..15
                  ((n * 37) % 256).astype(np.uint8)[:, None]):  # full uint8, incl. > 128
        p = problem("int4", 65536, 32, packed, scales, zeros, group=32)
        _, ref = oracle.dequant(packed, scales, zeros, "int4", 32)
        assert_bits_equal(gpu_dequant_bits(p), ref, "int4 exhaustive")


@pytest.mark.parametrize("group", [32, 64, 128, 256])
def test_dequant_int4_groups(group):
    packed, scales, zeros = synth.make_weights("int4", 64, 1024, group=group, seed=group)
    p = problem("int4", 64, 1024, packed, scales, zeros, group=group)
    _, ref = oracle.dequant(packed, scales, zeros, "int4", group)
    assert_bits_equal(gpu_dequant_bits(p), ref, f"int4 g{group}")


def test_dequant_writes_only_its_output():
    import weight_only_bit_w4a16_gb300 as wq
    packed, scales, zeros = synth.make_weights("int4", 5, 256, seed=2)
    p = problem("int4", 5, 256, packed, scales, zeros)
    _, pk, sc, zr = to_dev(dict(p, A=np.zeros((1, 256), np.uint16)))
    buf = torch.full((5 * 256 + 64,), -7.0, dtype=torch.bfloat16, device="cuda")
    W = buf[: 5 * 256].view(5, 256)
    wq.dequant(pk, sc, zr, "int4", out=W)
    torch.cuda.synchronize()
    assert torch.all(buf[5 * 256:] == -7.0)
    _, ref = oracle.dequant(packed, scales, zeros, "int4", 128)
    assert_bits_equal(W.view(torch.int16).cpu().numpy().view(np.uint16), ref, "guarded")
