"""Pins of the oracle's prepacked layout (CPU only).

The layout is a build-step repack that the KBench megakernel_int4_weight_decode
spec allows ("The weight format": interleaved nibbles, fragment pre-swizzle,
scales in a separate stream); its definition stands above wq_prepack_bytes in
include/wq.h.  oracle.prepack writes it with per-word loops; here it is held
to (1) hand-worked byte positions (tests/golden/prepack_examples.txt) and
(2) an inverse written independently (array reshapes and an inverse
permutation, bf16 decoded by PyTorch), under which every input bit comes back.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import prepack as opk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prepack_examples.txt")
GROUP = {"int4": 128, "nvfp4": 16, "mxfp4": 32}


def parse_golden():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        t = line.split()
        if t[0] == "case":
            cur = {"name": t[1], "fmt": t[2], "set": [], "expect": []}
        elif t[0] == "end":
            cases.append(cur)
            cur = None
        elif t[0] == "expect":
            cur["expect"].append((int(t[1], 0), int(t[2], 0)))
        else:
            cur["set"].append((t[0], int(t[1], 0), int(t[2], 0), int(t[3], 0)))
    return cases


def empty_weight(fmt, N=20, K=256):
    g = GROUP[fmt]
    packed = np.zeros((N, K // 2), np.uint8)
    if fmt == "int4":
        return packed, np.zeros((N, K // g), np.uint16), np.zeros((N, K // g), np.uint8)
    return packed, np.zeros((N, K // g), np.uint8), None


@pytest.mark.parametrize("case", parse_golden(), ids=lambda c: c["name"])
def test_hand_worked_positions(case):
    fmt = case["fmt"]
    packed, scales, zeros = empty_weight(fmt)
    for kind, row, col, val in case["set"]:
        if kind == "code":
            sh = 4 * (col & 1)
            byte = int(packed[row, col // 2])
            packed[row, col // 2] = (byte & (0xFF ^ (0xF << sh))) | (val << sh)
        elif kind == "scale":
            scales[row, col] = val
        else:
            zeros[row, col] = val
    buf = opk.prepack(packed, scales, zeros, fmt, GROUP[fmt])
    assert buf.size == opk.prepack_bytes(20, 256, fmt)
    for off, byte in case["expect"]:
        assert buf[off] == byte, (case["name"], off, hex(buf[off]), hex(byte))
    # the code region holds nothing but the codes that were set
    ncode = 2 * 2 * 1024
    nset = sum(1 for s in case["set"] if s[0] == "code" and s[3] != 0)
    assert np.count_nonzero(buf[:ncode]) <= nset


def test_sizes():
    # Nb * I * (1024 + record block) (+ 16 flag bytes for int4): 20 rows -> 2
    # blocks, K 256 -> 2 blocks
    assert opk.prepack_bytes(20, 256, "int4") == 4 * (1024 + 48) + 16
    assert opk.prepack_bytes(20, 256, "nvfp4") == 4 * (1024 + 128)
    assert opk.prepack_bytes(20, 256, "mxfp4") == 4 * (1024 + 64)
    assert opk.prepack_bytes(16, 128, "int4") == 1024 + 48 + 16
    assert opk.prepack_bytes(8192, 3072, "int4") == 512 * 24 * 1072 + 16


# -- an independent inverse ----------------------------------------------------
STORED_WORD = np.array([0, 4, 1, 5, 2, 6, 3, 7])     # stored slot q holds word STORED_WORD[q]
INT4_NIBBLE_OF_K = np.array([0, 4, 1, 5, 2, 6, 3, 7])  # int4: k0 + t sits in nibble INT4_NIBBLE_OF_K[t]


def bf16_value(bits):
    a = np.asarray(bits, np.uint16).astype(np.int16)
    return torch.from_numpy(a.copy()).view(torch.bfloat16).to(torch.float64).numpy()


def unprepack(buf, N, K, fmt):
    nb, nk = -(-N // 16), -(-K // 128)
    code = buf[:nb * nk * 1024].reshape(nb, nk, 2, 16, 2, 16)          # b i h r chunk byte
    swapped = ((np.arange(16) >> 2) & 1) == 1
    logical = code.copy()
    logical[:, :, :, swapped] = code[:, :, :, swapped][:, :, :, :, ::-1]
    stored = logical.reshape(nb, nk, 2, 16, 8, 4)                       # b i h r slot byte
    words = np.empty_like(stored)
    words[:, :, :, :, STORED_WORD] = stored                             # b i h r u byte
    nib = np.stack([words & 0xF, words >> 4], axis=-1).reshape(nb, nk, 2, 16, 8, 8)
    if fmt == "int4":
        nib = nib[..., INT4_NIBBLE_OF_K]                                # -> k order
    codes = nib.transpose(0, 3, 1, 2, 4, 5).reshape(nb * 16, nk * 128)  # (row, k)
    codes = codes[:N, :K]
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)

    rec = buf[nb * nk * 1024:]
    if fmt == "int4":
        blocks = rec[:nb * nk * 48].reshape(nb, nk, 48)
        sc = blocks[:, :, :32].reshape(nb, nk, 8, 2, 2)                       # b i (r&7) (r>>3) bytes
        sc = sc.transpose(0, 3, 2, 1, 4).reshape(nb * 16, nk, 2)              # row i bytes
        zp = blocks[:, :, 32:].reshape(nb, nk, 8, 2).transpose(0, 3, 2, 1).reshape(nb * 16, nk)
        s_bits = sc[..., 0].astype(np.uint16) | (sc[..., 1].astype(np.uint16) << 8)
        flags = rec[nb * nk * 48:]
        return packed, s_bits[:N], zp[:N], (s_bits[N:], zp[N:], flags)
    per = 8 if fmt == "nvfp4" else 4
    blocks = rec.reshape(nb, nk, 16, per).transpose(0, 2, 1, 3).reshape(nb * 16, nk * per)
    ng = K // GROUP[fmt]
    return packed, blocks[:N, :ng], None, (blocks[N:], blocks[:N, ng:])


@pytest.mark.parametrize("fmt,N,K", [
    ("int4", 16, 128), ("int4", 37, 384), ("int4", 64, 1024),
    ("nvfp4", 16, 128), ("nvfp4", 33, 160), ("nvfp4", 48, 544),
    ("mxfp4", 5, 96), ("mxfp4", 40, 416),
])
def test_round_trip(fmt, N, K):
    rng = np.random.default_rng(N * 1000 + K)
    g = GROUP[fmt]
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    if fmt == "int4":
        scales = rng.integers(0, 1 << 16, (N, K // g), dtype=np.uint16)
        zeros = rng.integers(0, 256, (N, K // g), dtype=np.uint8)     # full uint8, > 128 included
    else:
        scales = rng.integers(0, 256, (N, K // g), dtype=np.uint8)
        zeros = None
    buf = opk.prepack(packed, scales, zeros, fmt, g)
    assert buf.size == opk.prepack_bytes(N, K, fmt)
    p2, s2, z2, pad = unprepack(buf, N, K, fmt)
    np.testing.assert_array_equal(p2, packed)
    if fmt == "int4":
        np.testing.assert_array_equal(s2, scales)
        np.testing.assert_array_equal(z2, zeros)
        s_pad, z_pad, flags = pad
        assert not s_pad.any() and not z_pad.any()
        assert flags.size == 16 and int(flags[0]) == int((zeros > 128).any()) and not flags[1:].any()
    else:
        np.testing.assert_array_equal(s2, scales)
        assert not pad[0].any() and not pad[1].any()
    # padding codes (rows past N, k past K) are 0: the code region holds
    # exactly as many nonzero nibbles as the input
    nb, nk = -(-N // 16), -(-K // 128)
    code = buf[:nb * nk * 1024]
    nz_in = np.count_nonzero(packed & 0xF) + np.count_nonzero(packed >> 4)
    nz_out = np.count_nonzero(code & 0xF) + np.count_nonzero(code >> 4)
    assert nz_in == nz_out


def test_large_zero_flag():
    """The int4 flag byte is 1 exactly when some zero point exceeds 128
    (128 itself is still one exact subtrahend)."""
    packed = np.zeros((20, 128), np.uint8)
    scales = np.zeros((20, 2), np.uint16)
    for zmax, want in ((0, 0), (128, 0), (129, 1), (255, 1)):
        zeros = np.zeros((20, 2), np.uint8)
        zeros[19, 1] = zmax
        buf = opk.prepack(packed, scales, zeros, "int4", 128)
        assert int(buf[4 * (1024 + 48)]) == want, zmax


def test_first_subtrahend_is_exact():
    # bf16(128 + min(z, 128)) and bf16(z - min(z, 128)) hold the zero point
    # exactly for every uint8 z (the decode's two subtrahends)
    for z in range(256):
        zc = min(z, 128)
        a, b = oracle.round_bf16(128.0 + zc), oracle.round_bf16(float(z - zc))
        assert bf16_value([a])[0] + bf16_value([b])[0] - 128.0 == z


def test_prepack_rejects_other_groups():
    packed = np.zeros((16, 128), np.uint8)
    with pytest.raises(ValueError):
        opk.prepack(packed, np.zeros((16, 4), np.uint16), np.zeros((16, 4), np.uint8), "int4", 64)
