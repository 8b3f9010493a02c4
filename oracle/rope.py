"""Rotary position embedding (oracle; test infrastructure only).

The pages describe a Llama-style block but do not print its RoPE.  Reading:
the Llama "rotate-half" pairing of channel i with i + d/2, inverse frequency
base^(-2i/d), applied to q and k at the new token's position before the
Hadamard rotation (RoPE in the model basis), with no frequency rescaling.
"""
import numpy as np


def inv_freq(head_dim: int, base: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / head_dim)


def rope_apply(x, pos: int, base: float) -> np.ndarray:
    """Rotate the last axis (head_dim) of x at integer position ``pos`` in FP64."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = float(pos) * inv_freq(d, base)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
