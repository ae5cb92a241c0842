"""Helpers of the GPU parity tests: device upload, the call through the C ABI,
and the element-wise comparison against the oracle.

The tolerance is the gate of the method: for fp32 output
|C_gpu - C_exact| <= 1e-3 * S + 1e-6 with S = sum_k |a_mk * w_nk|, and bf16
output adds 2^-8 * |C_exact| for the final rounding (oracle.tolerance).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import weight_only_bit_w4a16_gb300 as wq


def device():
    return torch.device("cuda:0")


def to_dev(p, dev=None):
    dev = dev or device()
    A = torch.from_numpy(p["A"].view(np.int16)).view(torch.bfloat16).to(dev)
    packed = torch.from_numpy(p["packed"]).to(dev)
    if p["fmt"] == "int4":
        scales = torch.from_numpy(p["scales"].view(np.int16)).view(torch.bfloat16).to(dev)
        zeros = torch.from_numpy(p["zeros"]).to(dev)
    else:
        scales = torch.from_numpy(p["scales"]).to(dev)
        zeros = None
    return A, packed, scales, zeros


def gpu_gemm_dev(p, out="bf16", path="auto", workspace=None):
    """C on the device (the whole output never crosses to the host)."""
    A, packed, scales, zeros = to_dev(p)
    C = wq.gemm(A, packed, scales, zeros, p["fmt"], p["group"], out_dtype=out, path=path, workspace=workspace)
    torch.cuda.synchronize()
    assert wq.wq_get_device_error() == wq.WQ_OK
    return C


def gpu_gemm(p, out="bf16", path="auto", workspace=None):
    return gpu_gemm_dev(p, out, path, workspace).float().cpu().numpy().astype(np.float64)


def host_rows_cols(C, rows, cols):
    """C[rows, :] and C[:, cols] of a device result, as float64 host arrays;
    only the sampled rows and columns are copied."""
    r = torch.from_numpy(rows).to(C.device)
    c = torch.from_numpy(cols).to(C.device)
    return (C.index_select(0, r).float().cpu().numpy().astype(np.float64),
            C.index_select(1, c).float().cpu().numpy().astype(np.float64))


def gpu_dequant_bits(p):
    _, packed, scales, zeros = to_dev(p)
    W = wq.dequant(packed, scales, zeros, p["fmt"], p["group"])
    torch.cuda.synchronize()
    return W.view(torch.int16).cpu().numpy().view(np.uint16)


def sample(n, k, seed):
    """Sorted distinct indices in [0, n): the ends plus k random ones."""
    rng = np.random.default_rng(seed)
    idx = set([0, n - 1]) | set(rng.integers(0, n, size=min(k, n)).tolist())
    return np.array(sorted(idx), dtype=np.int64)


def oracle_ref(p, rows=None, cols=None):
    return oracle.gemm(p["A"], p["packed"], p["scales"], p["zeros"], p["fmt"], p["group"], rows, cols)


def assert_parity(C, Ce, S, out, what=""):
    tol = oracle.tolerance(Ce, S, out)
    err = np.abs(C - Ce)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - tol, -np.inf)), C.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{C.size} outside the gate; worst at {i}: "
            f"gpu={C[i]!r} exact={Ce[i]!r} tol={tol[i]!r}")


def check_full(p, out, path="auto", what="", workspace=None):
    C = gpu_gemm(p, out, path, workspace)
    Ce, S = oracle_ref(p)
    assert_parity(C, Ce, S, out, what)
    return C


def check_sampled(p, out, path="auto", k=24, seed=0, what="", workspace=None):
    """Full GPU result; oracle on sampled rows (all columns) and sampled
    columns (all rows), only those copied to the host."""
    C = gpu_gemm_dev(p, out, path, workspace)
    M, N = C.shape
    rows = sample(M, k, seed)
    cols = sample(N, k, seed + 1)
    Cr, Cc = host_rows_cols(C, rows, cols)
    del C
    Ce, S = oracle_ref(p, rows=rows)
    assert_parity(Cr, Ce, S, out, what + " rows")
    Ce, S = oracle_ref(p, cols=cols)
    assert_parity(Cc, Ce, S, out, what + " cols")
