"""Algorithmic bytes and flops of one call (the roofline numerators).

Bytes are what the method must move at least once: A (M x K bf16), the packed
codes (N x K/2), the scales (1 byte per group for the fp4 formats, 2 for the
int4 bf16 scale) and the int4 zero points (1 byte per group), and C (M x N,
2 or 4 bytes).  Flops are 2 M N K; the method saves bytes, not flops.
The KBench megakernel_int4_weight_decode.py spec prices a decode step of the
3B model the same way (its "bytes_per_step", and "The LM head is 197 MB
packed" in its performance notes); tests/test_metrics.py reproduces both.
"""
from __future__ import annotations

SCALE_BYTES = {"nvfp4": 1, "mxfp4": 1, "int4": 2}


def weight_bytes(fmt: str, N: int, K: int, group: int) -> int:
    g = N * (K // group)
    return N * K // 2 + g * SCALE_BYTES[fmt] + (g if fmt == "int4" else 0)


def call_bytes(fmt: str, M: int, N: int, K: int, group: int, out: str = "bf16") -> int:
    return 2 * M * K + weight_bytes(fmt, N, K, group) + M * N * (4 if out == "fp32" else 2)


def call_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
