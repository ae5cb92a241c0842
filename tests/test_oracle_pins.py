"""Pins of the oracle to things other than itself (CPU only).

Each test checks the oracle against a value fixed by the pages or by the
mathematics: hand-worked bytes (tests/golden/decode_examples.txt), exhaustive
decodes against PyTorch's own float8 / bfloat16 casts, exact rational dot
products, exact invariants, and "mutation" checks that show the tolerance
gate rejects the known ways of getting the decode wrong (the failure modes
listed in the Precision section of the KBench megakernel_int4_weight_decode
spec, plus the missing-subnormal e2m1 decode of the TileLang example's
_tir_u8_to_f4_to_bf16).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from weight_only_bit_w4a16_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "decode_examples.txt")


# -- independent decoders (library casts / textbook formulas, test-only) ----
def ind_e4m3(b):
    t = torch.tensor(np.array(b, dtype=np.uint8).reshape(-1)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy().reshape(np.shape(b))


def ind_bf16(bits):
    a = np.array(bits, dtype=np.uint16).reshape(-1).view(np.int16)
    t = torch.from_numpy(a.copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy().reshape(np.shape(bits))


def ind_e8m0(b):
    b = np.array(b, dtype=np.int64)
    if hasattr(torch, "float8_e8m0fnu"):
        t = torch.tensor(b.astype(np.uint8).reshape(-1)).view(torch.float8_e8m0fnu)
        return t.to(torch.float64).numpy().reshape(b.shape)
    out = np.ldexp(1.0, b - 127)
    return np.where(b == 255, np.nan, out)


def ind_e2m1(code):
    """Textbook e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa, subnormal at e=0."""
    code = np.asarray(code, dtype=np.int64)
    s = np.where(code & 8, -1.0, 1.0)
    e = (code >> 1) & 3
    m = code & 1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, e - 1))
    return s * mag


def ind_dequant(packed, scales, zeros, fmt, group):
    """Test-only vectorised decode built from the independent decoders."""
    N, Kh = packed.shape
    K = 2 * Kh
    codes = np.empty((N, K), dtype=np.int64)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    g = np.arange(K) // group
    if fmt == "nvfp4":
        return ind_e2m1(codes) * np.abs(ind_e4m3(scales))[:, g]
    if fmt == "mxfp4":
        return ind_e2m1(codes) * ind_e8m0(scales)[:, g]
    # An infinite scale times a zero offset is NaN, the same as the oracle's IEEE product.
    with np.errstate(invalid="ignore"):
        return (codes - zeros.astype(np.int64)[:, g]) * ind_bf16(scales)[:, g]


def bf16_of_exact(x):
    """RNE bf16 of fp64 values that are exact in fp32 (true for int4 weights):
    fp64 -> fp32 is exact, fp32 -> bf16 is torch's RNE cast."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.float32)
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def same_values(a, b):
    """Exact equality including the sign of zero; NaN matches NaN."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nan = np.isnan(a) | np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return np.all(np.where(nan, np.isnan(a) & np.isnan(b), eq))


def is_bf16_nan(bits):
    bits = np.asarray(bits, dtype=np.int64)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x7F) != 0)


# -- golden hand-worked bytes -------------------------------------------------
def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            fmt, byte, scale, zero, kp, value, bits = line.split()
            rows.append((fmt, int(byte, 16), int(scale, 16),
                         0 if zero == "-" else int(zero), int(kp),
                         float(value), int(bits, 16)))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: f"{r[0]}-{r[1]:#04x}-{r[2]:#x}-k{r[4]}")
def test_golden_decode(row):
    fmt, byte, scale, zero, kp, value, bits = row
    group = synth.GROUP[fmt]
    K = group                       # one group, the byte sits at k = 0, 1
    packed = np.zeros((1, K // 2), dtype=np.uint8)
    packed[0, 0] = byte
    sdt = np.uint16 if fmt == "int4" else np.uint8
    scales = np.array([[scale]], dtype=sdt)
    zeros = np.array([[zero]], dtype=np.uint8) if fmt == "int4" else None
    w = oracle.weight(packed, scales, zeros, fmt, group, 0, kp)
    assert same_values(w, value), (w, value)
    W64, Wb = oracle.dequant(packed, scales, zeros, fmt, group)
    assert same_values(W64[0, kp], value)
    if math.isnan(value):
        assert is_bf16_nan(Wb[0, kp])
    else:
        assert int(Wb[0, kp]) == bits, (hex(int(Wb[0, kp])), hex(bits))


def test_golden_file_has_every_format():
    fmts = {r[0] for r in _golden_rows()}
    assert fmts == {"nvfp4", "mxfp4", "int4"}


# -- exhaustive scalar decoders against library casts ------------------------
def test_e2m1_table_matches_textbook_formula():
    for c in range(16):
        assert same_values(oracle.e2m1(c), ind_e2m1(c)), c
    # the value set of the e2m1 grid: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}
    assert sorted({abs(oracle.e2m1(c)) for c in range(16)}) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_all_256_bytes_match_torch():
    ref = ind_e4m3(np.arange(256))
    got = np.array([oracle.e4m3(b) for b in range(256)])
    assert same_values(got, ref)
    assert oracle.e4m3(0x7E) == 448.0 and oracle.e4m3(0x08) == 2.0 ** -6
    assert oracle.e4m3(0x07) == 0.013671875 and oracle.e4m3(0x01) == 2.0 ** -9
    assert np.isnan(oracle.e4m3(0x7F)) and np.isnan(oracle.e4m3(0xFF))


def test_e8m0_all_256_bytes():
    ref = ind_e8m0(np.arange(256))
    got = np.array([oracle.e8m0(b) for b in range(256)])
    assert same_values(got, ref)
    assert oracle.e8m0(127) == 1.0 and oracle.e8m0(0) == 2.0 ** -127


def test_bf16_all_65536_patterns_match_torch():
    bits = np.arange(65536)
    ref = ind_bf16(bits)
    got = np.array([oracle.bf16(int(b)) for b in bits])
    assert same_values(got, ref)


def test_round_bf16_matches_torch_on_fp32_grid():
    # every bf16 high half with low halves that hit ties, near-ties and carries
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    u = (hi[:, None] | lows[None, :]).reshape(-1)
    f32 = u.view(np.float32)
    ref = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16(float(x)) for x in f32], dtype=np.uint16)
    nan = np.isnan(f32)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(is_bf16_nan(got[nan]))


def test_round_bf16_rounds_the_exact_fp64_value():
    one = 0x3F80
    assert oracle.round_bf16(1 + 2.0 ** -8) == one              # tie -> even (down)
    assert oracle.round_bf16(1 + 3 * 2.0 ** -8) == one + 2      # tie -> even (up)
    assert oracle.round_bf16(1 + 2.0 ** -8 + 2.0 ** -40) == one + 1
    assert oracle.round_bf16(1 + 2.0 ** -8 - 2.0 ** -40) == one
    # a value whose fp32 image is a tie: rounding through fp32 would give 0x3F80
    assert oracle.round_bf16(1 + 2.0 ** -8 + 2.0 ** -30) == one + 1
    assert oracle.round_bf16(-0.0) == 0x8000
    assert oracle.round_bf16(3.5e38) == 0x7F80                  # above bf16 max + half ulp
    assert oracle.round_bf16(2.0 ** -134) == 0x0000             # half the min subnormal: tie -> 0
    assert oracle.round_bf16(2.0 ** -134 * 1.0000001) == 0x0001
    assert oracle.round_bf16(1e300) == 0x7F80 and oracle.round_bf16(-1e300) == 0xFF80


# -- whole-array decode against the independent decoder ----------------------
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
def test_dequant_matches_independent_decode_random(fmt):
    packed, scales, zeros = synth.make_weights(fmt, 64, 512, seed=3)
    W64, Wb = oracle.dequant(packed, scales, zeros, fmt, synth.GROUP[fmt])
    ref = ind_dequant(packed, scales, zeros, fmt, synth.GROUP[fmt])
    assert same_values(W64, ref)
    assert np.array_equal(Wb, bf16_of_exact(ref))


def test_dequant_fp4_every_code_with_every_scale_byte():
    # row b uses scale byte b; the row's 32 codes run 0..15 twice
    codes = np.tile(np.arange(16), 2)
    row = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    packed = np.tile(row, (256, 1))
    for fmt in ("nvfp4", "mxfp4"):
        group = synth.GROUP[fmt]
        scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 32 // group, axis=1)
        W64, Wb = oracle.dequant(packed, scales, None, fmt, group)
        ref = ind_dequant(packed, scales, None, fmt, group)
        assert same_values(W64, ref), fmt
        fin = np.isfinite(ref)
        # fp4 weights have at most 6 significant bits: exact in fp32, and the
        # bf16 image is the value itself unless it leaves the bf16 range
        assert np.array_equal(Wb[fin], bf16_of_exact(ref[fin])), fmt
        assert np.all(is_bf16_nan(Wb[np.isnan(ref)])), fmt


def test_dequant_int4_every_bf16_scale_code_and_zero():
    # row n uses scale bits n and zero n % 16; its 32 codes run 0..15 twice
    n = np.arange(65536)
    codes = np.tile(np.arange(16), 2)
    row = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    packed = np.tile(row, (65536, 1))
    scales = n.astype(np.uint16)[:, None]
    zeros = (n % 16).astype(np.uint8)[:, None]
    W64, Wb = oracle.dequant(packed, scales, zeros, "int4", 32)
    ref = ind_dequant(packed, scales, zeros, "int4", 32)
    assert same_values(W64, ref)
    nan = np.isnan(ref)
    assert np.array_equal(Wb[~nan], bf16_of_exact(ref[~nan]))
    assert np.all(is_bf16_nan(Wb[nan]))
    # full uint8 zero points (beyond the promised 0..15) are read as they are
    zeros2 = ((n * 37) % 256).astype(np.uint8)[:, None]
    W2, _ = oracle.dequant(packed[:4096], scales[:4096], zeros2[:4096], "int4", 32)
    assert same_values(W2, ind_dequant(packed[:4096], scales[:4096], zeros2[:4096], "int4", 32))


# -- nibble order ------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
def test_nibble_order_low_nibble_is_even_k(fmt):
    group = synth.GROUP[fmt]
    K = group
    packed = np.zeros((1, K // 2), dtype=np.uint8)
    packed[0, 0] = 0x10                   # k=0 -> code 0, k=1 -> code 1
    if fmt == "int4":
        scales = np.array([[0x3F80]], dtype=np.uint16)    # 1.0
        zeros = np.array([[0]], dtype=np.uint8)
        expect = {0: 0.0, 1: 1.0}
    else:
        scales = np.array([[0x38 if fmt == "nvfp4" else 127]], dtype=np.uint8)  # 1.0
        zeros = None
        expect = {0: 0.0, 1: 0.5}
    for k, v in expect.items():
        A = np.zeros((1, K), dtype=np.uint16)
        A[0, k] = 0x3F80                  # one-hot activation at k
        C, S = oracle.gemm(A, packed, scales, zeros, fmt, group)
        assert C[0, 0] == v and S[0, 0] == abs(v)


# -- brute force with exact rationals ----------------------------------------
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
@pytest.mark.parametrize("groups", [1, 2])
def test_gemm_brute_force_fractions(fmt, groups):
    group = synth.GROUP[fmt]
    M, N, K = 3, 4, groups * group
    p = synth.make_problem(fmt, M, N, K, seed=11 + groups)
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], fmt, group)
    a = ind_bf16(p["A"])
    w = ind_dequant(p["packed"], p["scales"], p["zeros"], fmt, group)
    for m in range(M):
        for n in range(N):
            exact = sum((Fraction(float(a[m, k])) * Fraction(float(w[n, k])) for k in range(K)),
                        Fraction(0))
            sabs = sum((abs(Fraction(float(a[m, k])) * Fraction(float(w[n, k]))) for k in range(K)),
                       Fraction(0))
            assert abs(Fraction(C[m, n]) - exact) <= Fraction(K) * Fraction(2) ** -52 * sabs
            assert abs(Fraction(S[m, n]) - sabs) <= Fraction(K) * Fraction(2) ** -52 * sabs


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
def test_gemm_matches_numpy_matmul_of_independent_decode(fmt):
    p = synth.make_problem(fmt, 8, 96, 1024, seed=5)
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    a = ind_bf16(p["A"])
    w = ind_dequant(p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    ref = a @ w.T
    sref = np.abs(a) @ np.abs(w).T
    bound = 1024 * 2.0 ** -52 * sref
    assert np.all(np.abs(C - ref) <= bound)
    assert np.all(np.abs(S - sref) <= bound)
    # row / column subsets give the same numbers as the full product
    rows, cols = np.array([7, 0, 3]), np.array([95, 10, 11, 0])
    Cs, Ss = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], fmt, p["group"], rows, cols)
    assert np.array_equal(Cs, C[np.ix_(rows, cols)]) and np.array_equal(Ss, S[np.ix_(rows, cols)])


# -- exact invariants ----------------------------------------------------------
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
def test_one_hot_activation_selects_a_weight(fmt):
    p = synth.make_problem(fmt, 1, 32, 256, seed=7)
    W64, _ = oracle.dequant(p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    ks = np.array([0, 1, 17, 128, 255])
    A = np.zeros((len(ks), 256), dtype=np.uint16)
    A[np.arange(len(ks)), ks] = 0x3F80
    C, _ = oracle.gemm(A, p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    assert np.array_equal(C, W64[:, ks].T)
    # identity activation: C = W^T
    I = np.zeros((256, 256), dtype=np.uint16)
    I[np.arange(256), np.arange(256)] = 0x3F80
    C, _ = oracle.gemm(I, p["packed"], p["scales"], p["zeros"], fmt, p["group"])
    assert np.array_equal(C, W64.T)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_fp4_sign_flip_negates_exactly(fmt):
    p = synth.make_problem(fmt, 4, 16, 256, seed=9)
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], None, fmt, p["group"])
    C2, S2 = oracle.gemm(p["A"], p["packed"] ^ 0x88, p["scales"], None, fmt, p["group"])
    assert np.array_equal(C2, -C) and np.array_equal(S2, S)


def test_mxfp4_exponent_plus_one_doubles_exactly():
    p = synth.make_problem("mxfp4", 4, 16, 256, seed=10)
    C, _ = oracle.gemm(p["A"], p["packed"], p["scales"], None, "mxfp4", 32)
    C2, _ = oracle.gemm(p["A"], p["packed"], p["scales"] + 1, None, "mxfp4", 32)
    assert np.array_equal(C2, 2 * C)


def test_int4_codes_equal_zero_point_give_zero():
    N, K, g = 8, 256, 128
    z = np.random.default_rng(1).integers(0, 16, size=(N, K // g), dtype=np.uint8)
    codes = np.repeat(z, g, axis=1)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = synth.bf16_bits(np.full((N, K // g), 0.01, np.float32))
    A = synth.draw_A(np.random.default_rng(2), 4, K)
    C, S = oracle.gemm(A, packed, scales, z, "int4", g)
    assert np.all(C == 0) and np.all(S == 0)


def test_nvfp4_zero_scale_gives_zero():
    p = synth.make_problem("nvfp4", 4, 8, 256, seed=4)
    C, S = oracle.gemm(p["A"], p["packed"], np.zeros_like(p["scales"]), None, "nvfp4", 16)
    assert np.all(C == 0) and np.all(S == 0)


# -- the gate has teeth: known wrong decodes fail it --------------------------
def _violations(C, Cref, S, out):
    tol = oracle.tolerance(Cref, S, out)
    return np.mean(np.abs(C - Cref) > tol)


@pytest.mark.parametrize("case", ["tiny_nvfp4", "decode_int4"])
def test_wrong_decodes_fail_the_gate(case):
    w = synth.WORKLOADS[case]
    M, N, K = (16, 256, 512) if case == "tiny_nvfp4" else (4, 256, 3072)
    p = synth.make_problem(w["fmt"], M, N, K, seed=0, scale_mult=w.get("scale_mult", 0.5))
    fmt, g, out = p["fmt"], p["group"], w["out"]
    args = (p["A"], p["packed"], p["scales"], p["zeros"], fmt, g)
    C, S = oracle.gemm(*args)
    assert _violations(C, C, S, out) == 0

    swapped = ((p["packed"] & 0xF) << 4 | (p["packed"] >> 4)).astype(np.uint8)
    C1, _ = oracle.gemm(p["A"], swapped, p["scales"], p["zeros"], fmt, g)
    assert _violations(C1, C, S, out) > 0.9, "nibbles read high-first"

    row_s = np.repeat(p["scales"][:, :1], p["scales"].shape[1], axis=1)
    row_z = None if p["zeros"] is None else np.repeat(p["zeros"][:, :1], p["zeros"].shape[1], axis=1)
    C2, _ = oracle.gemm(p["A"], p["packed"], row_s, row_z, fmt, g)
    assert _violations(C2, C, S, out) > 0.9, "one (scale, zero) per row"

    if fmt == "int4":
        C3, _ = oracle.gemm(p["A"], p["packed"], p["scales"], np.zeros_like(p["zeros"]), fmt, g)
        assert _violations(C3, C, S, out) > 0.9, "zero point ignored"
    else:
        # the TileLang helper's decode: exponent field 0 read as a normal
        # number, so code 0 -> 0.5 and code 1 -> 0.75 (times the scale)
        W64, _ = oracle.dequant(p["packed"], p["scales"], None, fmt, g)
        codes = np.empty((N, K), dtype=np.int64)
        codes[:, 0::2] = p["packed"] & 0xF
        codes[:, 1::2] = p["packed"] >> 4
        scale = np.abs(ind_e4m3(p["scales"]))[:, np.arange(K) // g]
        Wm = W64.copy()
        for c, v in ((0, 0.5), (1, 0.75), (8, -0.5), (9, -0.75)):
            Wm[codes == c] = v * scale[codes == c]
        C4 = ind_bf16(p["A"]) @ Wm.T
        assert _violations(C4, C, S, out) > 0.5, "e2m1 subnormals decoded as normals"
