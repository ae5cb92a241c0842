"""The prepacked weight layout, written out byte by byte from its definition.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing in the product
library imports this module, and it shares no code with the library's repack
kernel.  The layout is a build-step choice the KBench spec leaves open (its
untimed build step may store the weights however the kernel likes best, for
example with nibbles interleaved, pre-arranged for the MMA fragments and the
scales in a stream of their own); its definition is the one stated above ``wq_prepack_bytes`` in ``include/wq.h``,
restated here:

* codes: ``Nb = ceil(N/16)`` row blocks x ``I = ceil(K/128)`` k-blocks of
  1024 bytes, block ``(b, i)`` at ``(b*I + i)*1024``.  Half ``h`` (k from
  ``128i + 64h``) at ``+512h``; row ``r`` of the half at ``32r``; the row's
  eight words ``w0..w7`` (``w_u`` = the 8 codes from ``k0 = 128i + 64h + 8u``)
  in the order ``w0 w4 w1 w5 | w2 w6 w3 w7``, the two 16-byte halves of the
  row exchanged when bit 2 of ``r`` is set.  fp4 words keep the input's byte
  order; int4 words hold ``k0 + 2s`` in nibble ``s`` and ``k0 + 2s + 1`` in
  nibble ``s + 4``.  Padding (rows past N, k past K): code 0.
* records from ``Nb*I*1024``, one per code block:
  int4 (group 128) 48 bytes: row r's bf16 scale at ``4*(r&7) + 2*(r>>3)``,
  its uint8 zero point at ``32 + 2*(r&7) + (r>>3)``; padded rows 0 and 0.
  NVFP4 128 bytes: row r's 8 scale bytes (groups ``8i..8i+7``) at ``8r``.
  MXFP4 64 bytes: row r's 4 scale bytes (groups ``4i..4i+3``) at ``4r``.
  Groups past K and padded rows: 0.
* int4 only, 16 bytes after the last record block: byte 0 is 1 when some
  zero point exceeds 128, else 0; the rest 0.
"""
from __future__ import annotations

import numpy as np


_INT4, _NVFP4, _MXFP4 = "int4", "nvfp4", "mxfp4"
_WORD_ORDER = (0, 4, 1, 5, 2, 6, 3, 7)   # storage order of a half-row's words


def _fmt_name(fmt) -> str:
    names = {0: _NVFP4, 1: _MXFP4, 2: _INT4}
    return names[fmt] if isinstance(fmt, int) else str(fmt)


def record_bytes(fmt) -> int:
    """Bytes of one record block."""
    return {_INT4: 48, _NVFP4: 128, _MXFP4: 64}[_fmt_name(fmt)]


def flag_bytes(fmt) -> int:
    """Bytes after the record blocks (int4: the large-zero-point flag)."""
    return 16 if _fmt_name(fmt) == _INT4 else 0


def prepack_bytes(N: int, K: int, fmt) -> int:
    nb, nk = -(-N // 16), -(-K // 128)
    return nb * nk * (1024 + record_bytes(fmt)) + flag_bytes(fmt)


def _codes(packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Code of every (row, k), zero beyond the weight: low nibble = even k."""
    N, half = packed.shape
    c = np.zeros((rows, cols), dtype=np.uint8)
    c[:N, 0:2 * half:2] = packed & 0x0F
    c[:N, 1:2 * half:2] = packed >> 4
    return c


def _word_bytes(eight_codes, fmt: str) -> list:
    """The 4 bytes of one word holding 8 codes of consecutive k."""
    c = [int(v) for v in eight_codes]
    if fmt == _INT4:
        nib = [c[0], c[2], c[4], c[6], c[1], c[3], c[5], c[7]]   # nibble s, s + 4
    else:
        nib = c                                                  # input order
    return [nib[2 * j] | (nib[2 * j + 1] << 4) for j in range(4)]


def prepack(packed, scales, zeros, fmt, group: int) -> np.ndarray:
    """The prepacked buffer (uint8, ``prepack_bytes`` long) of one weight."""
    fmt = _fmt_name(fmt)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N, half = packed.shape
    K = 2 * half
    if fmt == _INT4 and group != 128 or fmt == _NVFP4 and group != 16 or fmt == _MXFP4 and group != 32:
        raise ValueError("prepack takes int4 group 128, nvfp4 group 16, mxfp4 group 32")
    nb, nk = -(-N // 16), -(-K // 128)
    codes = _codes(packed, nb * 16, nk * 128)
    out = np.zeros(prepack_bytes(N, K, fmt), dtype=np.uint8)

    # ---- code blocks
    for b in range(nb):
        for i in range(nk):
            blk = (b * nk + i) * 1024
            for h in range(2):
                for r in range(16):
                    row = 16 * b + r
                    words = []
                    for u in range(8):
                        k0 = 128 * i + 64 * h + 8 * u
                        words.append(_word_bytes(codes[row, k0:k0 + 8], fmt))
                    logical = []
                    for u in _WORD_ORDER:
                        logical += words[u]
                    if (r >> 2) & 1:
                        logical = logical[16:] + logical[:16]
                    at = blk + 512 * h + 32 * r
                    out[at:at + 32] = logical

    # ---- record blocks
    rec0 = nb * nk * 1024
    rb = record_bytes(fmt)
    if fmt == _INT4:
        s_bits = np.asarray(scales, dtype=np.uint16)
        z_all = np.asarray(zeros, dtype=np.uint8)
    else:
        s_all = np.asarray(scales, dtype=np.uint8)
    ng = K // group
    for b in range(nb):
        for i in range(nk):
            at = rec0 + (b * nk + i) * rb
            for r in range(16):
                row = 16 * b + r
                if fmt == _INT4:
                    if row < N:
                        s, z = int(s_bits[row, i]), int(z_all[row, i])
                    else:
                        s, z = 0, 0
                    p = at + 4 * (r & 7) + 2 * (r >> 3)
                    out[p:p + 2] = [s & 0xFF, s >> 8]
                    out[at + 32 + 2 * (r & 7) + (r >> 3)] = z
                else:
                    per = 8 if fmt == _NVFP4 else 4
                    for g in range(per):
                        gi = per * i + g
                        if row < N and gi < ng:
                            out[at + per * r + g] = s_all[row, gi]
    if fmt == _INT4 and N > 0 and bool((z_all > 128).any()):
        out[rec0 + nb * nk * rb] = 1
    return out
