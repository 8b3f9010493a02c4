"""Block-diagonal Hadamard rotation (oracle; test infrastructure only).

The summary page ("무엇과 다른가") applies a block-diagonal Hadamard transform
to K and V before cache quantisation, and the same transform to the query and
(inverted) to the attention output, so that q^T k is preserved.  The pages do
not say which Hadamard; the reading taken is the normalised Sylvester matrix
in natural order, H[i, j] = (-1)^popcount(i & j) / sqrt(n), which is symmetric
and orthogonal, hence its own inverse.
"""
import numpy as np


def sylvester(n: int) -> np.ndarray:
    """Normalised Sylvester-Hadamard matrix of order n (a power of two), FP64."""
    if n < 1 or n & (n - 1):
        raise ValueError("order must be a power of two")
    i = np.arange(n)
    par = np.zeros((n, n), dtype=np.int64)
    m = i[:, None] & i[None, :]
    while np.any(m):
        par ^= m & 1
        m = m >> 1
    return np.where(par == 1, -1.0, 1.0) / np.sqrt(n)


def blockdiag_apply(x, block: int) -> np.ndarray:
    """Apply H_block to each consecutive block of the last axis of x (FP64)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    if d % block:
        raise ValueError("last axis must be a multiple of the block")
    h = sylvester(block)
    xb = x.reshape(x.shape[:-1] + (d // block, block))
    return (xb @ h.T).reshape(x.shape)
