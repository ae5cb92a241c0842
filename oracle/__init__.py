"""The oracle: a plain, slow fp64 CPU implementation of C = A . deq(B)^T.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s ``cpu_baseline`` / ``--impl reference`` leg may import this
package.  The product library under ``weight_only_bit_w4a16_gb300/`` never
imports it, and the two share no code, header, table or constant.

The arithmetic lives in ``wq_oracle.c`` (plain C, fp64, bit-by-bit decoders,
an explicit e2m1 table, a plain k-ascending dot product).  This module only
builds that file with gcc, loads it with ctypes and marshals numpy arrays.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
fixed by the pages and by the mathematics (hand-worked bytes, exhaustive
decodes against independent decoders, exact rational dot products, exact
invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libwq_oracle.so")

#: format codes of the oracle's own C interface
FORMATS = {"nvfp4": 0, "mxfp4": 1, "int4": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile wq_oracle.c into a shared library (gcc, fp64, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-std=c99", "-Wall", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            d, i, vp = ctypes.c_double, ctypes.c_int, ctypes.c_void_p
            L.wqo_e2m1.restype = d; L.wqo_e2m1.argtypes = [i]
            L.wqo_e4m3.restype = d; L.wqo_e4m3.argtypes = [i]
            L.wqo_e8m0.restype = d; L.wqo_e8m0.argtypes = [i]
            L.wqo_bf16.restype = d; L.wqo_bf16.argtypes = [i]
            L.wqo_round_bf16.restype = i; L.wqo_round_bf16.argtypes = [d]
            L.wqo_weight.restype = d
            L.wqo_weight.argtypes = [vp, vp, vp, i, i, i, i, i, i]
            L.wqo_dequant.restype = None
            L.wqo_dequant.argtypes = [vp, vp, vp, i, i, i, i, vp, vp]
            L.wqo_gemm.restype = None
            L.wqo_gemm.argtypes = [vp, vp, vp, vp, i, i, i, i, i,
                                   vp, i, vp, i, vp, vp]
            L.wqo_max_threads.restype = i; L.wqo_max_threads.argtypes = []
            L.wqo_set_threads.restype = None; L.wqo_set_threads.argtypes = [i]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


# -- scalar decoders (exposed for the pins) ----------------------------------
def e2m1(code: int) -> float:
    return lib().wqo_e2m1(int(code))


def e4m3(byte: int) -> float:
    return lib().wqo_e4m3(int(byte))


def e8m0(byte: int) -> float:
    return lib().wqo_e8m0(int(byte))


def bf16(bits: int) -> float:
    return lib().wqo_bf16(int(bits))


def round_bf16(x: float) -> int:
    """bf16 bits of x rounded to nearest even (uint16 value)."""
    return lib().wqo_round_bf16(float(x)) & 0xFFFF


# -- array entry points -------------------------------------------------------
def _check(packed, scales, zeros, fmt, group):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N, Kh = packed.shape
    K = 2 * Kh
    f = _fmt(fmt)
    sdt = np.uint16 if f == FORMATS["int4"] else np.uint8
    scales = np.ascontiguousarray(scales, dtype=sdt)
    assert scales.shape == (N, K // group), (scales.shape, N, K, group)
    if f == FORMATS["int4"]:
        zeros = np.ascontiguousarray(zeros, dtype=np.uint8)
        assert zeros.shape == (N, K // group)
    else:
        zeros = None
    return packed, scales, zeros, N, K, f


def weight(packed, scales, zeros, fmt, group, n, k) -> float:
    packed, scales, zeros, N, K, f = _check(packed, scales, zeros, fmt, group)
    return lib().wqo_weight(_ptr(packed), _ptr(scales), _ptr(zeros), N, K, f,
                            int(group), int(n), int(k))


def dequant(packed, scales, zeros, fmt, group):
    """Return (W64, Wbf16): exact fp64 weights and their RNE bf16 bits, (N, K)."""
    packed, scales, zeros, N, K, f = _check(packed, scales, zeros, fmt, group)
    W64 = np.empty((N, K), dtype=np.float64)
    Wb = np.empty((N, K), dtype=np.uint16)
    lib().wqo_dequant(_ptr(packed), _ptr(scales), _ptr(zeros), N, K, f,
                      int(group), _ptr(W64), _ptr(Wb))
    return W64, Wb


def gemm(A_bits, packed, scales, zeros, fmt, group, rows=None, cols=None):
    """Return (C, S): the exact fp64 product and the tolerance scale.

    A_bits is the (M, K) bf16 activation as uint16 bits.  ``rows`` / ``cols``
    select a subset of output rows (m) / columns (n); None means all.
    """
    packed, scales, zeros, N, K, f = _check(packed, scales, zeros, fmt, group)
    A_bits = np.ascontiguousarray(A_bits, dtype=np.uint16)
    M = A_bits.shape[0]
    assert A_bits.shape == (M, K)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int32)
    nr = M if r is None else len(r)
    nc = N if c is None else len(c)
    if r is not None:
        assert r.size == 0 or (r.min() >= 0 and r.max() < M)
    if c is not None:
        assert c.size == 0 or (c.min() >= 0 and c.max() < N)
    C = np.zeros((nr, nc), dtype=np.float64)
    S = np.zeros((nr, nc), dtype=np.float64)
    if nr and nc and K:
        lib().wqo_gemm(_ptr(A_bits), _ptr(packed), _ptr(scales), _ptr(zeros),
                       M, N, K, f, int(group), _ptr(r), nr, _ptr(c), nc,
                       _ptr(C), _ptr(S))
    return C, S


def tolerance(C_exact, S, out_dtype: str):
    """Allowed |C_gpu - C_exact| per element.

    fp32 output: 1e-3 * S + 1e-6; bf16 output adds 2^-8 * |C_exact| for the
    final rounding of the output.
    """
    tol = 1e-3 * np.asarray(S) + 1e-6
    if out_dtype == "bf16":
        tol = tol + np.abs(np.asarray(C_exact)) * 2.0 ** -8
    return tol


def max_threads() -> int:
    return lib().wqo_max_threads()


def set_threads(n: int) -> None:
    lib().wqo_set_threads(int(n))


# ---------------------------------------------------------------------------
# Fused epilogues (bias, the SiLU-gated product of a gate/up projection pair,
# residual; the KBench spec's decoder MLP).  Plain fp64 definitions on
# top of the exact product above; no arithmetic is shared with the library.
# ---------------------------------------------------------------------------
def silu(x):
    """SiLU(x) = x * sigmoid(x) = x / (1 + e^-x), in fp64 (KBench spec's decoder
    MLP: down(silu(gate(x)) * up(x)))."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def bf16_array(bits):
    """bf16 bit patterns -> fp64 values, element by element through the
    bit-by-bit decoder."""
    bits = np.asarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    flat_in, flat_out = bits.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = bf16(int(flat_in[i]))
    return out


def gated_rows(n_weight_rows: int):
    """Weight-row indices (gate, up) of each gated output column.  The gate
    and up rows of one output come in interleaved groups of 8: weight rows
    16b .. 16b+7 are the gate rows of outputs 8b .. 8b+7 and rows 16b+8 ..
    16b+15 their up rows."""
    assert n_weight_rows % 16 == 0
    o = np.arange(n_weight_rows // 2)
    gate = 16 * (o // 8) + (o % 8)
    return gate, gate + 8


def epilogue(C, S, bias_bits=None, residual_bits=None, gated=False, out_dtype="fp32"):
    """Apply the fused epilogue to the exact product C (M, N weight rows) and
    return (Y, T): the exact fp64 result and the allowed |Y_gpu - Y| per element.

        y = C + bias[n]                      (bias: bf16 per weight row)
        gated: y_o = silu(y_gate(o)) * y_up(o)  (gated_rows)
        y += residual[m, o]                  (residual: bf16, (M, outputs))

    The tolerance carries the product's gate (1e-3 S + 1e-6, fp32
    accumulation) through the epilogue: each weight row's value may be off by
    e = 1e-3 S + 1e-6 + 2^-22 |y|; silu has slope at most 1.0999 (its
    derivative sigmoid(x) (1 + x (1 - sigmoid(x))) peaks there), so the gated
    value may be off by 1.1 |u| e_g + (|silu(g)| + 1.1 e_g) e_u; the fp32
    arithmetic of the epilogue adds 2^-19 |y|, and bf16 output 2^-8 |y|.
    """
    C = np.asarray(C, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    y = C.copy()
    if bias_bits is not None:
        y = y + bf16_array(bias_bits)[None, :]
    e = 1e-3 * S + 1e-6 + 2.0 ** -22 * np.abs(y)
    if gated:
        gi, ui = gated_rows(C.shape[1])
        g, u, eg, eu = y[:, gi], y[:, ui], e[:, gi], e[:, ui]
        sg = silu(g)
        y = sg * u
        t = 1.1 * np.abs(u) * eg + (np.abs(sg) + 1.1 * eg) * eu
    else:
        t = e
    if residual_bits is not None:
        y = y + bf16_array(residual_bits)
    t = t + 2.0 ** -19 * np.abs(y) + 1e-6
    if out_dtype == "bf16":
        t = t + 2.0 ** -8 * np.abs(y)
    return y, t
