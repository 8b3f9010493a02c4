"""Symmetric INT4 group quantiser (oracle; test infrastructure only).

Follows the summary page, "무엇과 다른가" (INT4 values, group scales applied
after accumulation, nibbles stored with an offset of 8) and "전제와 한계"
(round-to-nearest weights).  Readings where the pages are silent:

* symmetric scale s = amax / 7, rounded to BF16 (ties to even);
* the code is c = clamp(rne(x / s), -8, 7) + 8 taken against the BF16 scale,
  so that decoding (c - 8) * s is self-consistent; an all-zero group has
  s = 0 and every code 8;
* every rounding decision (amax / 7, x / s, rne) is taken in FP32, the
  precision the kernels decide in, so both sides reach the same integers.
"""
import numpy as np

from .numerics import bf16_rne, bf16_from_bits


def quantize_groups(x, group: int):
    """Quantise the last axis of FP32 ``x`` in consecutive groups of ``group``.

    Returns (codes uint8 in [0, 15], scales FP32 holding BF16 values) with
    scales shaped [..., n // group].
    """
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[-1]
    if n % group:
        raise ValueError("last axis must be a multiple of the group size")
    xg = x.reshape(x.shape[:-1] + (n // group, group))
    amax = np.max(np.abs(xg), axis=-1)
    s = bf16_rne(amax / np.float32(7.0))
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    t = (xg / safe[..., None]).astype(np.float32)
    q = np.clip(np.rint(t), -8, 7)
    q = np.where((s == 0)[..., None], 0.0, q)
    codes = (q + 8).astype(np.uint8).reshape(x.shape)
    return codes, s.astype(np.float32)


def dequantize_groups(codes, scales, group: int) -> np.ndarray:
    """x_hat = (c - 8) * s in FP64 (the group scale applied to each group)."""
    c = np.asarray(codes).astype(np.float64) - 8.0
    n = c.shape[-1]
    cg = c.reshape(c.shape[:-1] + (n // group, group))
    return (cg * np.asarray(scales, dtype=np.float64)[..., None]).reshape(c.shape)


def nibble_decode_via_bf16(code: int) -> float:
    """Value of nibble ``code`` by the pages' construction: place the nibble in
    the mantissa of BF16 128.0 (bit pattern 0x4300) and subtract 136
    (summary page, "무엇과 다른가").  Used only to pin the offset-8 reading."""
    v = float(bf16_from_bits(np.array([0x4300 | (int(code) & 0xF)], dtype=np.uint16))[0])
    return v - 136.0
