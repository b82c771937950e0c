"""Tensor fusion: one contiguous buffer holding many small gradient tensors.

DisCo, Introduction (tensor fusion): several small gradient tensors are fused
into one before the AllReduce, and the fused tensor's size is the sum of the
small ones' sizes.  Readings where the page is silent: tensors are placed in
index order, each starting at a 256-byte aligned byte offset; the bytes
between tensors and after the last one (up to the rounded total) are zero;
the fused values are x * scale rounded to float32, then to bfloat16 with
round-to-nearest-even; unpacking widens bfloat16 to float32 exactly and
multiplies by ``uscale`` (float32).
"""
from __future__ import annotations

import numpy as np


def align_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def layout(numels, elem_bytes=2, align=256):
    """Byte offset of every tensor and the buffer's total size."""
    offs, cur = [], 0
    for n in numels:
        offs.append(cur)
        cur = align_up(cur + int(n) * elem_bytes, align)
    return offs, cur


def bf16_rne_bits(x):
    """float32 -> bfloat16 bit patterns, IEEE-754 round to nearest, ties to even.

    The bfloat16 value is the upper half of a float32.  Adding 0x7FFF plus the
    lowest kept bit to the float32 bits and keeping the upper 16 bits rounds
    to nearest with ties to even; a carry out of the mantissa correctly bumps
    the exponent, and values beyond the largest finite bfloat16 become
    infinity.  NaN maps to the quiet NaN 0x7FC0 with its sign.
    """
    b = np.asarray(x, dtype=np.float32).reshape(-1).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    isnan = ((b & np.uint64(0x7F800000)) == np.uint64(0x7F800000)) & ((b & np.uint64(0x007FFFFF)) != 0)
    r = np.where(isnan, (b >> np.uint64(16)) & np.uint64(0x8000) | np.uint64(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _scaled(x, scale):
    return (np.asarray(x, dtype=np.float32).astype(np.float64) * np.float64(np.float32(scale))).astype(np.float32)


def pack(tensors, scale, buf_dtype="bf16", align=256):
    """Fusion buffer as a uint8 array."""
    eb = 2 if buf_dtype == "bf16" else 4
    offs, total = layout([t.size for t in tensors], eb, align)
    buf = np.zeros(total, dtype=np.uint8)
    for t, o in zip(tensors, offs):
        y = _scaled(t.reshape(-1), scale)
        data = bf16_rne_bits(y).view(np.uint8) if eb == 2 else y.view(np.uint8)
        buf[o:o + data.size] = data
    return buf


def unpack(buf, numels, uscale, buf_dtype="bf16", align=256):
    """Float32 tensors recovered from the fusion buffer."""
    eb = 2 if buf_dtype == "bf16" else 4
    offs, _ = layout(numels, eb, align)
    out = []
    for n, o in zip(numels, offs):
        raw = buf[o:o + int(n) * eb]
        x = bf16_bits_to_f32(raw.view(np.uint16)) if eb == 2 else raw.view(np.float32)
        out.append(_scaled(x, uscale))
    return out
