"""Pins of the parity gate itself (CPU only).

Every GPU parity test compares against oracle.tolerance (the product) or the
T of oracle.epilogue (fused epilogues), so their values are pinned here to
numbers worked by hand from the stated gate:

  fp32 output  |C_gpu - C_exact| <= 1e-3 * S + 1e-6,   S = sum_k |a_ik w_jk|
  bf16 output  the same + 2^-8 * |C_exact|             (the output rounding)

(the benchmark spec of the method's tolerance; the KBench spec's
Precision section describes the gate as an arithmetic bound, not an
exactness check).  A slip in either constant, a dropped absolute term, or
the bf16 term applied to fp32 output fails one of these.
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import oracle  # noqa: E402
from gpu_util import assert_parity  # noqa: E402


# (S, C_exact, output, allowed error), each worked by hand
GATE_CASES = [
    (1000.0, 0.0, "fp32", 1.000001),        # 1e-3 * 1000 + 1e-6
    (0.0, 256.0, "fp32", 0.000001),         # no output-rounding term for fp32
    (0.0, 256.0, "bf16", 1.000001),         # 1e-6 + 256 / 256
    (1000.0, -512.0, "bf16", 3.000001),     # 1 + 1e-6 + 512 / 256
    (0.0, 0.0, "fp32", 0.000001),           # the absolute floor alone
    (0.0, 0.0, "bf16", 0.000001),
    (2.5e5, 3.0, "bf16", 250.011719750),    # 250 + 1e-6 + 3 / 256 = 250.01171875 + 1e-6
]


@pytest.mark.parametrize("S,C,out,want", GATE_CASES)
def test_gate_values_by_hand(S, C, out, want):
    got = float(oracle.tolerance(np.array([C]), np.array([S]), out)[0])
    assert abs(got - want) <= 1e-12 * max(1.0, want), (got, want)


def test_gate_broadcasts_elementwise():
    S = np.array([[1000.0, 0.0], [1000.0, 0.0]])
    C = np.array([[0.0, 256.0], [-512.0, 256.0]])
    got = oracle.tolerance(C, S, "bf16")
    want = np.array([[1.000001, 1.000001], [3.000001, 1.000001]])
    assert np.allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("out,S,C,tol", [("fp32", 1000.0, 0.0, 1.000001), ("bf16", 0.0, 256.0, 1.000001)])
def test_just_inside_and_just_outside(out, S, C, tol):
    """The parity helper every GPU test uses accepts an error just inside the
    gate and rejects one just outside it."""
    Ce, Se = np.array([[C]]), np.array([[S]])
    assert_parity(np.array([[C + tol * (1 - 1e-9)]]), Ce, Se, out, "inside")
    assert_parity(np.array([[C - tol * (1 - 1e-9)]]), Ce, Se, out, "inside, below")
    with pytest.raises(AssertionError):
        assert_parity(np.array([[C + tol * (1 + 1e-6)]]), Ce, Se, out, "outside")


# ---- the fused epilogue's T ----------------------------------------------------
# Its rule (the oracle's docstring and the design notes): each weight row's
# value may be off by e = 1e-3 S + 1e-6 + 2^-22 |y|; the gated value by
# 1.1 |u| e_g + (|silu(g)| + 1.1 e_g) e_u; the epilogue's fp32 arithmetic
# adds 2^-19 |y| + 1e-6, bf16 output 2^-8 |y|.

def bf16(x):
    return np.array([np.frombuffer(np.float32(x).tobytes(), np.uint16)[1]], dtype=np.uint16)


def test_epilogue_tolerance_by_hand_ungated():
    """C = 2, S = 100, bias 0.5, residual -1 (all exact in bf16), one element:
      y before the residual = 2.5;  e = 0.1 + 1e-6 + 2.5 * 2^-22
                                       = 0.100001596046447754
      y = 1.5;  T = e + 1.5 * 2^-19 + 1e-6 = 0.100005457069396973 (fp32 out)
      bf16 out: T + 1.5 / 256 = 0.105864832069396973."""
    C, S = np.array([[2.0]]), np.array([[100.0]])
    y, t = oracle.epilogue(C, S, bf16(0.5), bf16(-1.0).reshape(1, 1), False, "fp32")
    assert y[0, 0] == 1.5
    assert abs(t[0, 0] - 0.100005457069396973) < 1e-15
    _, tb = oracle.epilogue(C, S, bf16(0.5), bf16(-1.0).reshape(1, 1), False, "bf16")
    assert abs(tb[0, 0] - 0.105864832069396973) < 1e-15


def test_epilogue_tolerance_by_hand_gated():
    """A gate/up pair (weight rows 0 and 8 of 16) with g = 1, u = 2, S = 10,
    no bias or residual, fp32 out:
      silu(1) = 1 / (1 + e^-1) = 0.731058578630004879
      y = 2 silu(1) = 1.462117157260009758
      e_g = 0.01 + 1e-6 + 2^-22 = 0.010001238418579102
      e_u = 0.01 + 1e-6 + 2 * 2^-22 = 0.010001476837158203
      T = 1.1 * 2 * e_g + (silu(1) + 1.1 e_g) e_u + 2^-19 y + 1e-6
        = 0.022002724520874023 + 0.007421524588862... + 2.788776e-6 + 1e-6
        = 0.029428208598633678."""
    C = np.zeros((1, 16))
    C[0, 0], C[0, 8] = 1.0, 2.0
    S = np.full((1, 16), 10.0)
    y, t = oracle.epilogue(C, S, None, None, True, "fp32")
    assert abs(y[0, 0] - 1.462117157260009758) < 1e-15
    assert abs(t[0, 0] - 0.029428208598633678) < 1e-15
