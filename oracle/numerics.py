"""BF16 round-to-nearest-even on FP32 values (oracle; test infrastructure only).

The pages store group scales in BF16 (summary page, "무엇과 다른가").  The
rounding mode is not stated; the reading taken is IEEE round-half-to-even.
"""
import numpy as np


def bf16_rne(x) -> np.ndarray:
    """Round FP32 values to the nearest BF16 value, ties to even; returns FP32."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (r.astype(np.uint32) << 16).view(np.float32)


def bf16_bits(x) -> np.ndarray:
    """BF16 bit pattern (uint16) of FP32 values that are already BF16-exact."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    if np.any(b & 0xFFFF):
        raise ValueError("value is not representable in BF16")
    return (b >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
