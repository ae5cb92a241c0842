"""Seeded synthetic inputs for the W4A16 dequantise-GEMM.

This module only DRAWS inputs: shapes, value distributions and seeds of the
workloads.  It holds none of the method's arithmetic (no decoding, no
product, no accumulation), so both the oracle's tests and the CUDA path can
use it without sharing any of the computation.  Rounding a drawn fp32 value
to a storage type (bf16 activations and scales, e4m3 scales) is done by
PyTorch's own CPU casts, which round to nearest even.

Workloads (the shapes of the pages' decode and prefill use):
  * tiny_nvfp4     M=16, N=256, K=512, NVFP4 (e4m3 scale per 16), fp32 out.
  * decode_int4    M in {1, 4, 16}, N=8192, K=3072, int4 g128, bf16 out --
                   the gate/up projection of the 3B decoder in the KBench
                   megakernel_int4_weight_decode.py spec, at batch <= 16.
  * prefill_mxfp4  M=2048, N=K=3072, MXFP4 (e8m0 scale per 32), bf16 out.
  * large_nvfp4    M=N=K=8192, NVFP4, bf16 out.
  * layer_sweep    int4 g128 projections of that decoder (q, k/v, o, gate/up,
                   down, tied LM head) at M in {1, 16, 128, 2048}.

Distributions: A ~ N(0,1) rounded to bf16; packed bytes uniform over 0..255
(so both nibbles are uniform over the 16 codes); NVFP4 scales |N(0,1)|*c
rounded to e4m3 (c = 0.5 for tiny_nvfp4, 1 for large_nvfp4); MXFP4 scale
bytes 127 + U{-3..1}; int4 scales U(0.005, 0.02) rounded to bf16 and zeros
U{0..15}.  Draw order per problem: A, packed, scales, zeros, from
numpy.random.default_rng(seed).
"""
from __future__ import annotations

import numpy as np
import torch

GROUP = {"nvfp4": 16, "mxfp4": 32, "int4": 128}

#: 3B decoder dimensions (KBench megakernel_int4_weight_decode.py, CFG)
DECODER = dict(d=3072, ffn=8192, n_q=24, n_kv=8, hd=128, vocab=128256)

LAYER_SHAPES = {  # name: (N = out features, K = in features)
    "q": (3072, 3072),
    "kv": (1024, 3072),
    "o": (3072, 3072),
    "gate_up": (8192, 3072),
    "down": (3072, 8192),
    "lm_head": (128256, 3072),
}

WORKLOADS = {
    "tiny_nvfp4": dict(fmt="nvfp4", Ms=(16,), N=256, K=512, out="fp32",
                       scale_mult=0.5),
    "decode_int4": dict(fmt="int4", Ms=(1, 4, 16), N=8192, K=3072, out="bf16"),
    "prefill_mxfp4": dict(fmt="mxfp4", Ms=(2048,), N=3072, K=3072, out="bf16"),
    "large_nvfp4": dict(fmt="nvfp4", Ms=(8192,), N=8192, K=8192, out="bf16",
                        scale_mult=1.0),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), torch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> float8_e4m3fn bytes (uint8), torch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def draw_A(rng, M: int, K: int) -> np.ndarray:
    return bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


def draw_packed(rng, N: int, K: int) -> np.ndarray:
    return rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)


def draw_scales(rng, fmt: str, N: int, K: int, group: int, scale_mult=0.5):
    G = K // group
    if fmt == "nvfp4":
        s = np.abs(rng.standard_normal((N, G), dtype=np.float32)) * np.float32(scale_mult)
        return e4m3_bits(s), None
    if fmt == "mxfp4":
        return (127 + rng.integers(-3, 2, size=(N, G))).astype(np.uint8), None
    if fmt == "int4":
        s = rng.uniform(0.005, 0.02, size=(N, G)).astype(np.float32)
        scales = bf16_bits(s)
        zeros = rng.integers(0, 16, size=(N, G), dtype=np.uint8)
        return scales, zeros
    raise ValueError(fmt)


def make_weights(fmt: str, N: int, K: int, group: int | None = None, seed: int = 0,
                 scale_mult: float = 0.5, rng=None):
    """packed (N, K/2) uint8, scales (N, K/group), zeros (N, K/group) or None."""
    group = group or GROUP[fmt]
    rng = rng if rng is not None else np.random.default_rng(seed)
    packed = draw_packed(rng, N, K)
    scales, zeros = draw_scales(rng, fmt, N, K, group, scale_mult)
    return packed, scales, zeros


def make_problem(fmt: str, M: int, N: int, K: int, group: int | None = None,
                 seed: int = 0, scale_mult: float = 0.5) -> dict:
    """One seeded problem: A bits (M, K) uint16 plus the quantised weight."""
    group = group or GROUP[fmt]
    rng = np.random.default_rng(seed)
    A = draw_A(rng, M, K)
    packed, scales, zeros = make_weights(fmt, N, K, group, scale_mult=scale_mult, rng=rng)
    return dict(fmt=fmt, group=group, M=M, N=N, K=K, A=A, packed=packed,
                scales=scales, zeros=zeros)


def workload_problem(name: str, M: int | None = None, seed: int = 0) -> dict:
    w = WORKLOADS[name]
    M = w["Ms"][0] if M is None else M
    p = make_problem(w["fmt"], M, w["N"], w["K"], seed=seed,
                     scale_mult=w.get("scale_mult", 0.5))
    p["out"] = w["out"]
    return p


def layer_problem(layer: str, M: int, seed: int = 0) -> dict:
    N, K = LAYER_SHAPES[layer]
    p = make_problem("int4", M, N, K, seed=seed)
    p["out"] = "bf16"
    return p
