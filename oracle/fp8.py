"""E4M3 decode weights (oracle; test infrastructure only).

Summary page, "전제와 한계": the decode weights may be E4M3 instead of INT4
(a 0.02 perplexity cost); the abstract page compares the INT4 decode path with
an FP8 one.  The format is the OCP 8-bit E4M3 ("FN") encoding: sign, 4
exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
subnormals 2^-6 * m/8; no infinities; S.1111.111 is NaN, so the largest
finite magnitude is 2^8 * 1.75 = 448.

Readings where the pages are silent:
* the same group structure as the INT4 weights: per (output row, 128
  consecutive inputs) one BF16 scale, s = bf16(amax / 448), so the group's
  largest magnitude maps to the largest code;
* codes = E4M3(w / s) rounded to nearest, ties to even (the even code has
  mantissa LSB 0), values beyond 448 in magnitude saturate to +-448; an
  all-zero group has s = 0 and every code 0x00;
* as for INT4, w' = w * gamma, amax / 448 and w / s are formed in FP32 (the
  precision the kernels decide in) before the rounding decision.
"""
import numpy as np

from .numerics import bf16_rne

E4M3_MAX = 448.0
W_GROUP = 128


def e4m3_decode(code) -> np.ndarray:
    """Value(s) of 8-bit E4M3 code(s), FP64 (NaN for the two NaN codes)."""
    c = np.asarray(code).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    sub = np.ldexp(m / 8.0, -6)                        # exponent field 0: 2^(1-7) * m/8
    nrm = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    val = sign * np.where(e == 0, sub, nrm)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


# the 127 non-negative finite values, ascending with the code (0x00 .. 0x7E)
_POS = e4m3_decode(np.arange(0x7F))


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code(s) of FP64 value(s): ties to the even code, |x| > 448
    saturates to +-448, the sign is kept (a negative value that rounds to zero
    gives 0x80); x is taken exactly (callers round to FP32 first)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS, a, side="left"), 0, 0x7E)      # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _POS[lo], _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(_POS[hi] == a, hi, code)                           # exact values
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)   # the sign is kept, zero included


def quantize_weight_e4m3(w, gamma=None, group: int = W_GROUP):
    """FP32 W [N_out, K_in] (+ optional gamma [K_in]) -> (codes [N, K] u8 E4M3, scales [N, K/group] f32)."""
    w = np.asarray(w, dtype=np.float32)
    if gamma is not None:
        w = (w * np.asarray(gamma, dtype=np.float32)[None, :]).astype(np.float32)
    n, k = w.shape
    wg = w.reshape(n, k // group, group)
    amax = np.max(np.abs(wg), axis=-1)
    s = bf16_rne(amax / np.float32(E4M3_MAX))
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    t = (wg / safe[..., None]).astype(np.float32)
    codes = e4m3_encode(t.astype(np.float64))
    codes = np.where((s == 0)[..., None], np.uint8(0), codes).astype(np.uint8)
    return codes.reshape(n, k), s.astype(np.float32)


def e4m3_matvec(codes, scales, x, group: int = W_GROUP, row_chunk: int = 2048) -> np.ndarray:
    """y[b, o] = sum_g s[o, g] * sum_{i in g} e4m3(codes[o, i]) * x[b, i], in FP64
    (the group scale after each group's partial sum, as for INT4)."""
    x = np.asarray(x, dtype=np.float64)
    squeeze = x.ndim == 1
    if squeeze:
        x = x[None, :]
    n, k = codes.shape
    ng = k // group
    xg = x.reshape(x.shape[0], ng, group)
    y = np.empty((x.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, row_chunk):
        r1 = min(n, r0 + row_chunk)
        c = e4m3_decode(codes[r0:r1]).reshape(r1 - r0, ng, group)
        part = np.matmul(c.transpose(1, 0, 2), xg.transpose(1, 2, 0))
        s = np.asarray(scales[r0:r1], dtype=np.float64)
        y[:, r0:r1] = np.sum(part * s.T[:, :, None], axis=0).T
    return y[0] if squeeze else y
