"""Pins of the oracle's fused epilogue (bias, the SiLU-gated product of an
interleaved gate/up pair, residual) against closed forms and an independent
restatement (sigmoid through tanh, numpy matmul of the pinned dequant)."""
import math

import numpy as np
import pytest

import oracle
from weight_only_bit_w4a16_gb300 import synth


def silu_tanh(x):
    # sigmoid(x) = (1 + tanh(x / 2)) / 2: a different route to the same function
    x = np.asarray(x, dtype=np.float64)
    return x * 0.5 * (1.0 + np.tanh(0.5 * x))


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert oracle.silu(1.0) == pytest.approx(0.7310585786300049, rel=1e-15)
    assert oracle.silu(-1.0) == pytest.approx(-0.2689414213699951, rel=1e-15)
    # sigmoid(ln 3) = 3/4 exactly
    assert oracle.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    assert oracle.silu(-math.log(3.0)) == pytest.approx(-0.25 * math.log(3.0), rel=1e-15)
    # tails: x for large x, 0 for very negative x
    assert oracle.silu(60.0) == pytest.approx(60.0, rel=1e-15)
    assert abs(oracle.silu(-60.0)) < 1e-24
    # the tanh form cancels (1 + tanh) deep in the negative tail: compare where
    # both forms keep full precision
    xs = np.linspace(-6, 20, 2601)
    assert np.allclose(oracle.silu(xs), silu_tanh(xs), rtol=1e-12, atol=0)


def test_silu_slope_bound_used_by_the_tolerance():
    # the tolerance assumes |silu'| <= 1.1; the maximum is 1.0998...
    x = np.linspace(-30, 30, 600001)
    d = np.gradient(oracle.silu(x), x)
    assert d.max() < 1.1 and d.max() > 1.09 and d.min() > -0.11


def test_gated_row_map():
    g, u = oracle.gated_rows(16)
    assert g.tolist() == list(range(8)) and u.tolist() == list(range(8, 16))
    g, u = oracle.gated_rows(48)
    assert g.tolist() == list(range(0, 8)) + list(range(16, 24)) + list(range(32, 40))
    assert (u - g == 8).all()


def test_epilogue_by_hand():
    C = np.zeros((2, 16))
    C[0, 3], C[0, 11] = 1.0, 2.0       # output 3 of row 0: gate 1, up 2
    C[1, 0], C[1, 8] = -1.0, 4.0       # output 0 of row 1: gate -1, up 4
    S = np.zeros_like(C)
    bias = np.full(16, 0x0000, dtype=np.uint16)
    bias[3] = 0x3F80                   # +1.0 on weight row 3 (a gate row)
    res = np.zeros((2, 8), dtype=np.uint16)
    res[1, 0] = 0x3F00                 # +0.5 on output (1, 0)
    Y, T = oracle.epilogue(C, S, bias, res, gated=True)
    assert Y.shape == (2, 8)
    assert Y[0, 3] == pytest.approx(oracle.silu(2.0) * 2.0, rel=1e-15)
    assert Y[1, 0] == pytest.approx(oracle.silu(-1.0) * 4.0 + 0.5, rel=1e-15)
    assert Y[0, 0] == 0.0 and Y[1, 1] == 0.0
    # plain: bias then residual, no activation
    Y2, _ = oracle.epilogue(C, S, bias, np.zeros((2, 16), dtype=np.uint16), gated=False)
    assert Y2[0, 3] == 2.0 and Y2[0, 11] == 2.0 and Y2[1, 0] == -1.0


def test_epilogue_mutations_are_caught():
    """Swapping gate and up, or adding the bias after the gating, changes
    the result by far more than the tolerance."""
    rng = np.random.default_rng(0)
    C = rng.normal(size=(4, 32)) * 3
    S = np.abs(C) * 0.0
    Y, T = oracle.epilogue(C, S, gated=True)
    g, u = oracle.gated_rows(32)
    swapped = oracle.silu(C[:, u]) * C[:, g]
    assert (np.abs(swapped - Y) > T).any()
    bias = np.full(32, 0x3F80, dtype=np.uint16)
    Yb, Tb = oracle.epilogue(C, S, bias, gated=True)
    late = oracle.silu(C[:, g]) * C[:, u] + 1.0
    assert (np.abs(late - Yb) > Tb).any()


def test_epilogue_against_an_independent_restatement():
    """gemm + epilogue vs numpy: A @ W64^T of the pinned dequant, then the
    tanh-form SiLU, element by element."""
    p = synth.make_problem("int4", 3, 32, 256, seed=4)
    C, S = oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], "int4", 128)
    W64, _ = oracle.dequant(p["packed"], p["scales"], p["zeros"], "int4", 128)
    A64 = oracle.bf16_array(p["A"])
    rng = np.random.default_rng(1)
    bias = synth.bf16_bits(rng.normal(size=32).astype(np.float32))
    res = synth.bf16_bits(rng.normal(size=(3, 16)).astype(np.float32))
    Y, T = oracle.epilogue(C, S, bias, res, gated=True)
    y = A64 @ W64.T + oracle.bf16_array(bias)[None, :]
    g, u = oracle.gated_rows(32)
    ref = silu_tanh(y[:, g]) * y[:, u] + oracle.bf16_array(res)
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    assert (T > 0).all()
